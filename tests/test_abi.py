"""The C-ABI library without a GPU: it loads, exports what the header
declares, its struct layouts match the binding, and the host-only sizing
call validates configurations."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def gp():
    lib = os.path.join(ROOT, "demand_paged_kv_gqa_b300", "libgrowpage.so")
    if not os.path.exists(lib):
        from demand_paged_kv_gqa_b300 import build
        build.build()
    from demand_paged_kv_gqa_b300 import growpage
    return growpage


def declared_functions():
    names = set()
    for f in os.listdir(INCLUDE):
        if f.endswith(".h"):
            src = open(os.path.join(INCLUDE, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(gp_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(gp):
    names = declared_functions()
    assert len(names) >= 16
    for n in names:
        assert hasattr(gp.lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", gp.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (gp_[a-z0-9_]+)\b", out))
    assert set(names) <= exported, set(names) - exported


def test_struct_layouts_match_header(gp):
    prog = r"""
#include <stdio.h>
#include <stddef.h>
#include "growpage.h"
#define F(S, f) printf(#S "." #f " %zu\n", offsetof(S, f))
int main(void) {
  printf("gp_config %zu\ngp_layout %zu\ngp_req_meta %zu\ngp_ctrl %zu\ngp_state_view %zu\n",
         sizeof(gp_config), sizeof(gp_layout), sizeof(gp_req_meta), sizeof(gp_ctrl),
         sizeof(gp_state_view));
  F(gp_config, beta_s); F(gp_config, rope_theta); F(gp_config, flags);
  F(gp_layout, page_bytes); F(gp_layout, block_width); F(gp_layout, num_workers);
  F(gp_req_meta, delta); F(gp_req_meta, n_starved);
  F(gp_ctrl, steps); F(gp_ctrl, moved_tokens); F(gp_ctrl, shrinks);
  F(gp_req_meta, n_shrinks); F(gp_state_view, tok_pos); F(gp_state_view, free_stack);
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        exe = os.path.join(d, "t")
        open(c, "w").write(prog)
        subprocess.run(["gcc", "-I", INCLUDE, c, "-o", exe], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(l.split() for l in lines if l.strip())
    assert int(got["gp_config"]) == ctypes.sizeof(gp.gp_config)
    assert int(got["gp_layout"]) == ctypes.sizeof(gp.gp_layout)
    assert int(got["gp_req_meta"]) == ctypes.sizeof(gp.gp_req_meta) == 64
    assert int(got["gp_ctrl"]) == ctypes.sizeof(gp.gp_ctrl)
    assert int(got["gp_state_view"]) == ctypes.sizeof(gp.gp_state_view)
    for key, val in got.items():
        if "." in key:
            s, f = key.split(".")
            assert getattr(getattr(gp, s), f).offset == int(val), key


def _cfg(gp, **kw):
    base = dict(num_layers=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                num_pages=64, max_requests=4, max_pages_per_req=16, dtype=gp.GP_DTYPE_BF16,
                max_seq_len=2048, rope_theta=10000.0)
    base.update(kw)
    return gp.make_config(**base)


def test_pool_bytes_host_only(gp):
    n1 = gp.pool_bytes(_cfg(gp))
    n2 = gp.pool_bytes(_cfg(gp, num_pages=128))
    page = 2 * 2 * 2 * 16 * 128 * 2        # L * Hk * (K,V) * P * d * bf16
    assert n2 - n1 >= 64 * page
    assert n1 % 256 == 0
    # full-KV mode needs no summary-score region
    assert gp.pool_bytes(_cfg(gp, mode=gp.GP_MODE_FULL_KV)) < n1


@pytest.mark.parametrize("bad", [
    dict(num_q_heads=6), dict(num_q_heads=16, num_kv_heads=2), dict(page_size=8),
    dict(head_dim=96), dict(head_dim=64), dict(top_p=0.0), dict(top_p=1.5),
    dict(beta_s=1.0), dict(max_prefix_len=24), dict(mode=7), dict(mode=6), dict(recent_window=-1),
    dict(page_size=512),
])
def test_pool_bytes_rejects_unsupported(gp, bad):
    with pytest.raises(gp.GrowPageError):
        gp.pool_bytes(_cfg(gp, **bad))


def test_null_arguments_are_rejected_without_gpu(gp):
    assert gp.lib.gp_pool_bytes(None, None) == gp.GP_ERR_INVALID
    assert gp.lib.gp_destroy_pool(None) == gp.GP_ERR_INVALID
    assert gp.lib.gp_decode_step(None, 0, 0, None, None, None, None, None) == gp.GP_ERR_INVALID
    assert gp.lib.gp_get_state(None, None) == gp.GP_ERR_INVALID
    assert gp.lib.gp_launch_count(None) == 0
