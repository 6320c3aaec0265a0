"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function the header declares, agrees with the binding on the config
struct layout, and rejects bad arguments before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

from sparse_moe_layer_experts_b300 import binding as B
from sparse_moe_layer_experts_b300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam_moe.h")


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(beam_moe_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for want in ("beam_moe_route", "beam_moe_forward", "beam_moe_workspace_size",
                 "beam_moe_quantize_nvfp4", "beam_moe_read_status", "beam_moe_status_string"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_cfg_struct_layout_matches_header(tmp_path):
    fields = [f[0] for f in B.beam_moe_cfg._fields_]
    src = tmp_path / "layout.c"
    body = "\n".join(
        f'printf("{f} %zu\\n", offsetof(beam_moe_cfg, {f}));' for f in fields)
    src.write_text(
        "#include <stdio.h>\n#include <stddef.h>\n#include \"beam_moe.h\"\n"
        "int main(void){" + body + 'printf("SIZE %zu\\n", sizeof(beam_moe_cfg)); return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    out = dict(line.split() for line in subprocess.check_output([str(exe)], text=True).splitlines())
    for f in fields:
        assert int(out[f]) == getattr(B.beam_moe_cfg, f).offset, f
    assert int(out["SIZE"]) == ctypes.sizeof(B.beam_moe_cfg)


def test_beam_defaults_and_workspace_size(L):
    c = B.beam_moe_cfg()
    B.beam_moe_cfg_init_beam(c)
    assert (c.hidden, c.inter, c.n_experts, c.n_groups, c.topk_groups, c.top_k) == \
        (5120, 2560, 256, 8, 4, 8)
    assert c.routed_scale == 2.5
    s32 = B.beam_moe_workspace_size(32, c)
    s64 = B.beam_moe_workspace_size(64, c)
    assert 0 < s32 < s64
    # x_perm (bf16) + h (bf16) + y (bf16) dominate: 8 rows per token
    assert s64 - s32 >= 32 * 8 * (5120 * 2 + 2560 * 2 + 5120 * 2)
    assert B.beam_moe_hostio_extra_bytes(32, c) >= 2 * 32 * 5120 * 2


@pytest.mark.parametrize("field,value", [
    ("hidden", 100), ("inter", 64), ("n_experts", 258), ("n_groups", 3),
    ("topk_groups", 9), ("top_k", 33), ("top_k", 0), ("wtype", 7)])
def test_invalid_configs_rejected_on_host(L, field, value):
    c = B.beam_moe_cfg()
    B.beam_moe_cfg_init_beam(c)
    setattr(c, field, value)
    assert B.beam_moe_workspace_size(8, c) == 0
    rc = B.beam_moe_forward(16, 16, 16, 16, 16, 8, c, 16, None)
    assert rc == B.BEAM_MOE_ERR_INVALID_ARG
    rc = B.beam_moe_route(16, 16, 8, c, 16, 16, None, None, None, None, None)
    assert rc == B.BEAM_MOE_ERR_INVALID_ARG


def test_group_limit_rejects_too_many_experts(L):
    c = B.make_cfg(256, 128, 32, 8, 1, 5)  # one kept group of 4 experts < top-5
    assert B.beam_moe_workspace_size(8, c) == 0


def test_argument_errors_before_any_launch(L):
    c = B.beam_moe_cfg()
    B.beam_moe_cfg_init_beam(c)
    before = B.beam_moe_launch_count()
    # T = 0 is a successful no-op
    assert B.beam_moe_forward(None, None, None, None, None, 0, c, None, None) == B.BEAM_MOE_OK
    # null pointers
    assert B.beam_moe_forward(None, 16, 16, 16, 16, 4, c, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    # misaligned pointer
    assert B.beam_moe_forward(18, 16, 16, 16, 16, 4, c, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    # no workspace
    assert B.beam_moe_forward(16, 16, 16, 16, 16, 4, c, 16, None) == B.BEAM_MOE_ERR_WORKSPACE
    # workspace too small
    c.workspace, c.workspace_bytes = 1 << 20, 1024
    assert B.beam_moe_forward(16, 16, 16, 16, 16, 4, c, 16, None) == B.BEAM_MOE_ERR_WORKSPACE
    # negative and oversized T
    assert B.beam_moe_forward(16, 16, 16, 16, 16, -1, c, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_route(16, 16, 1 << 30, c, 16, 16, None, None, None, None,
                            None) == B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_launch_count() == before


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert B.beam_moe_status_string(code) != "unknown status"
    assert B.beam_moe_status_string(12345) == "unknown status"


def test_dense_entry_point_checks(L):
    c = B.beam_moe_cfg()
    c.hidden, c.inter, c.wtype = 256, 384, B.BEAM_MOE_W_BF16
    assert B.beam_moe_dense_workspace_size(64, c) > 64 * 384 * 2
    before = B.beam_moe_launch_count()
    assert B.beam_moe_dense_forward(None, None, None, None, 0, c, None, None) == B.BEAM_MOE_OK
    assert B.beam_moe_dense_forward(16, 16, 16, 16, 4, c, 16, None) == B.BEAM_MOE_ERR_WORKSPACE
    assert B.beam_moe_dense_forward(18, 16, 16, 16, 4, c, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    c.inter = 100
    assert B.beam_moe_dense_forward(16, 16, 16, 16, 4, c, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    c.inter, c.wtype = 384, B.BEAM_MOE_W_NVFP4
    assert B.beam_moe_dense_forward(16, 16, 16, 16, 4, c, 16, None) == B.BEAM_MOE_ERR_UNSUPPORTED
    assert B.beam_moe_dense_workspace_size(64, c) == 0
    assert B.beam_moe_launch_count() == before


def test_block_entry_point_checks(L):
    c = B.make_cfg(256, 128, 32, 8, 4, 8)
    assert B.beam_moe_block_workspace_size(64, c) > B.beam_moe_workspace_size(64, c)
    before = B.beam_moe_launch_count()
    assert B.beam_moe_block_forward(16, 9, 16, 16, 1e-6, 16, 16, 16, 16, 0, c, 16, None) == B.BEAM_MOE_OK
    assert B.beam_moe_block_forward(16, 0, 16, 16, 1e-6, 16, 16, 16, 16, 4, c, 16, None) == \
        B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_block_forward(16, 9, 16, 16, -1.0, 16, 16, 16, 16, 4, c, 16, None) == \
        B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_block_forward(16, 9, 16, 16, 1e-6, 16, 16, 16, 16, 4, c, 16, None) == \
        B.BEAM_MOE_ERR_WORKSPACE
    # quantised experts are accepted, but need their scale pointers
    for wt in (B.BEAM_MOE_W_NVFP4, B.BEAM_MOE_W_MXFP8):
        c.wtype = wt
        c.w_gate_sf = c.w_up_sf = c.w_down_sf = None
        assert B.beam_moe_block_forward(16, 9, 16, 16, 1e-6, 16, 16, 16, 16, 4, c, 16, None) == \
            B.BEAM_MOE_ERR_INVALID_ARG
        c.w_gate_sf = c.w_up_sf = c.w_down_sf = 16
        c.w_gate_gs = c.w_up_gs = c.w_down_gs = 16
        assert B.beam_moe_block_forward(16, 9, 16, 16, 1e-6, 16, 16, 16, 16, 4, c, 16, None) == \
            B.BEAM_MOE_ERR_WORKSPACE
    c.hidden = 8192 + 128
    assert B.beam_moe_block_forward(16, 9, 16, 16, 1e-6, 16, 16, 16, 16, 4, c, 16, None) == \
        B.BEAM_MOE_ERR_UNSUPPORTED
    assert B.beam_moe_launch_count() == before



def test_activation_quantiser_checks(L):
    before = B.beam_moe_launch_count()
    nv, mx = B.BEAM_MOE_W_NVFP4, B.BEAM_MOE_W_MXFP8
    assert B.beam_moe_quantize_act(nv, 16, 0, 64, 16, 16, None) == B.BEAM_MOE_OK
    assert B.beam_moe_quantize_act(B.BEAM_MOE_W_BF16, 16, 4, 64, 16, 16, None) == \
        B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_quantize_act(nv, 16, 4, 40, 16, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_quantize_act(mx, 16, 4, 48, 16, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_quantize_act(nv, 16, -1, 64, 16, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_quantize_act(nv, 18, 4, 64, 16, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_quantize_act(nv, None, 4, 64, 16, 16, None) == B.BEAM_MOE_ERR_INVALID_ARG
    assert B.beam_moe_launch_count() == before


def test_router_arith_by_batch_size():
    # Small batches keep the sequential FP32 FMA-chain router; from 256 tokens
    # the tensor-core router runs, and its split router weight (three bf16
    # parts of [E,H]) is carved from the workspace.
    c = B.beam_moe_cfg()
    B.beam_moe_cfg_init_beam(c)
    assert B.beam_moe_router_arith(1, c) == B.BEAM_MOE_ROUTER_FMA_CHAIN
    assert B.beam_moe_router_arith(255, c) == B.BEAM_MOE_ROUTER_FMA_CHAIN
    assert B.beam_moe_router_arith(256, c) == B.BEAM_MOE_ROUTER_TENSOR
    assert B.beam_moe_router_arith(1 << 20, c) == B.BEAM_MOE_ROUTER_TENSOR
    assert B.beam_moe_router_arith(-1, c) == B.BEAM_MOE_ERR_INVALID_ARG
    grow = B.beam_moe_workspace_size(256, c) - B.beam_moe_workspace_size(255, c)
    assert grow >= 3 * c.n_experts * c.hidden * 2
    c.top_k = 0
    assert B.beam_moe_router_arith(256, c) == B.BEAM_MOE_ERR_INVALID_ARG
