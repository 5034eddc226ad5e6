"""The C-ABI library loads without a GPU, exports every entry point that
include/moe_vq2.h declares, and rejects bad arguments on the host (these
calls return before any CUDA work is enqueued)."""
import ctypes
import os
import re

import pytest

import bit_vq_routed_gb300 as bv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_vq2.h")


def declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return bv.load()


def test_header_declares_expected_api():
    names = declared()
    for n in ["moe_route_topk", "moe_permute", "moe_vq2_expert_ffn", "moe_combine", "moe_slot_table_create",
              "moe_slot_table_set", "moe_router_logits"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(bv.EXPORTED) == set(declared())


def test_version_and_error_string(lib):
    assert lib.moe_version() >= 1
    assert isinstance(lib.moe_last_error(), bytes)


def _err(lib):
    return lib.moe_last_error().decode()


def test_router_rejects_bad_shapes(lib):
    P = ctypes.c_void_p
    assert lib.moe_router_logits(P(16), P(16), None, P(16), 1, 100, 8, None) == bv.MOE_ERR_UNSUPPORTED
    assert "256" in _err(lib)
    assert lib.moe_router_logits(None, P(16), None, P(16), 1, 256, 8, None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_router_logits(P(16), P(16), None, P(16), -1, 256, 8, None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_router_logits(P(18), P(16), None, P(16), 1, 256, 8, None) == bv.MOE_ERR_UNSUPPORTED
    # T = 0 is a no-op
    assert lib.moe_router_logits(None, None, None, None, 0, 256, 8, None) == bv.MOE_OK


def test_topk_rejects_bad_k(lib):
    P = ctypes.c_void_p
    assert lib.moe_route_topk(P(16), 4, 8, 0, 1, P(16), P(16), None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk(P(16), 4, 8, 9, 1, P(16), P(16), None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk(P(16), 4, 64, 33, 1, P(16), P(16), None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk(P(16), 4, 2048, 8, 1, P(16), P(16), None) == bv.MOE_ERR_UNSUPPORTED
    assert lib.moe_route_topk(P(16), 4, 8, 2, 7, P(16), P(16), None) == bv.MOE_ERR_INVALID_ARG


def test_permute_and_pack_reject_bad_args(lib):
    P = ctypes.c_void_p
    assert lib.moe_permute(P(16), 4, 2, 2000, P(16), P(16), P(16), None, 0, None) == bv.MOE_ERR_UNSUPPORTED
    assert lib.moe_permute(P(16), 4, 0, 8, P(16), P(16), P(16), None, 0, None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_vq2_pack(P(16), P(16), 15, 128, P(16), P(16), None) == bv.MOE_ERR_UNSUPPORTED
    assert lib.moe_vq2_pack(P(16), P(16), 16, 96, P(16), P(16), None) == bv.MOE_ERR_UNSUPPORTED
    assert lib.moe_fp4_pack(P(16), P(16), 16, 32, P(16), P(16), None) == bv.MOE_ERR_UNSUPPORTED
    assert lib.moe_fp4_pack(None, P(16), 16, 64, P(16), P(16), None) == bv.MOE_ERR_INVALID_ARG


def test_slot_table_and_ffn_reject_bad_args(lib):
    P = ctypes.c_void_p
    h = P()
    assert lib.moe_slot_table_create(8, 100, 128, P(16), ctypes.byref(h)) == bv.MOE_ERR_UNSUPPORTED
    assert h.value is None
    assert lib.moe_slot_table_create(0, 256, 128, P(16), ctypes.byref(h)) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_slot_table_create(8, 256, 128, None, ctypes.byref(h)) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_slot_table_set(None, 0, None, None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_slot_table_destroy(None) == bv.MOE_OK
    assert lib.moe_vq2_expert_ffn(None, P(16), P(16), P(16), P(16), 1, 8, 1, P(16), P(16), P(16), 1 << 20,
                                  None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(P(16), P(16), P(16), P(16), 2, 2, 256, None, None, None) == bv.MOE_ERR_INVALID_ARG


def test_workspace_sizes(lib):
    n = lib.moe_vq2_expert_ffn_workspace_size(1, 8, 256, 4096, 2048)
    assert n >= 8 * 2048 * 4
    assert lib.moe_vq2_expert_ffn_workspace_size(4096, 8, 256, 4096, 2048) >= 32768 * 2048 * 4
    # decode batch 32 at top-8 fits the scratch-free variant's fixed scratch
    assert lib.moe_vq2_expert_ffn_workspace_size(32, 8, 256, 4096, 2048) <= bv.MOE_NOALLOC_SCRATCH_BYTES
    # the permutation needs no workspace below 8192 pairs; from there two int32
    # per (1024-pair chunk, expert), after the routing counter's 256 bytes
    assert lib.moe_permute_workspace_size(1023, 8, 256) == 0
    assert lib.moe_permute_workspace_size(4096, 8, 256) == 2 * 4 * 32 * 256
    assert lib.moe_route_workspace_size(4096, 8, 256) == 256 + 2 * 4 * 32 * 256
    assert lib.moe_route_workspace_size(1, 8, 256) == 256


def test_launch_count_ignores_rejected_calls(lib):
    # calls that fail their host-side checks enqueue no kernel
    P = ctypes.c_void_p
    before = bv.moe_launch_count()
    assert lib.moe_router_logits(P(16), P(16), None, P(16), 1, 100, 8, None) == bv.MOE_ERR_UNSUPPORTED
    assert lib.moe_route_topk(P(16), 4, 8, 0, 1, P(16), P(16), None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_router_logits(None, None, None, None, 0, 256, 8, None) == bv.MOE_OK
    assert bv.moe_launch_count() == before


def test_route_rejects_bad_args(lib):
    P = ctypes.c_void_p
    assert lib.moe_route_workspace_size(1, 8, 256) >= 4
    args = [P(16), P(16), None, 1, 256, 8, 2, 1, P(16), P(16), P(16), P(16), P(16), P(16), P(16), 256, None]
    bad_k = list(args)
    bad_k[6] = 0
    assert lib.moe_route(*bad_k) == bv.MOE_ERR_INVALID_ARG
    bad_h = list(args)
    bad_h[4] = 100
    assert lib.moe_route(*bad_h) == bv.MOE_ERR_UNSUPPORTED
    no_ws = list(args)
    no_ws[14], no_ws[15] = None, 0
    assert lib.moe_route(*no_ws) == bv.MOE_ERR_WORKSPACE
    null_x = list(args)
    null_x[0] = None
    assert lib.moe_route(*null_x) == bv.MOE_ERR_INVALID_ARG


def test_header_compiles_as_plain_c(tmp_path):
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    src = tmp_path / "use_header.c"
    src.write_text('#include "moe_vq2.h"\nint main(void) { return moe_version() > 0 ? 0 : 1; }\n')
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I",
                        os.path.dirname(HEADER), "-I", cuda_inc, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_expert_cache_rejects_bad_args(lib):
    # host-side checks before any table is touched (no GPU needed)
    P = ctypes.c_void_p
    h = P(12345)
    assert lib.moe_expert_cache_create(None, P(256), 1 << 24, 6_684_672, ctypes.byref(h)) == bv.MOE_ERR_INVALID_ARG
    assert h.value is None  # the out handle is cleared first
    assert lib.moe_expert_cache_create(P(16), None, 1 << 24, 6_684_672, ctypes.byref(h)) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_cache_create(None, None, 0, 0, None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_cache_set_host(None, 0, None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_cache_set_host_image(None, 0, 0, P(16)) == bv.MOE_ERR_INVALID_ARG
    nf = ctypes.c_int(-1)
    assert lib.moe_expert_cache_fetch(None, None, 0, None, ctypes.byref(nf), None, None) == bv.MOE_ERR_INVALID_ARG
    assert lib.moe_expert_cache_slot_of(None, 0) == -1
    assert lib.moe_expert_cache_stats(None, None, None, None, None) == bv.MOE_ERR_INVALID_ARG
    assert "moe_expert_cache_stats" in lib.moe_last_error().decode()
    assert lib.moe_expert_cache_destroy(None, None) == bv.MOE_OK
