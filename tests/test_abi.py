"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/moe_gb300.h declares, and rejects bad arguments
with status codes before anything is launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")
PKG = os.path.join(ROOT, "mixture_experts_grouped_router_gb300")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__._build_module().build()
    from mixture_experts_grouped_router_gb300 import _lib
    return _lib


def test_header_declares_the_six_calls():
    names = _declared()
    for n in ("moe_route_topk", "moe_permute", "moe_gmm", "moe_tgmm", "moe_combine",
              "moe_unpermute_bwd", "moe_route_topk_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    lib = ctypes.CDLL(L._build.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_declared()) <= set(L.EXPORTED) | set(_declared())


def test_size_queries(L):
    assert L.moe_rows_cap(32768, 64, 1, 128) == 32768 + 64 * 127
    assert L.moe_rows_cap(100, 8, 2, 0) == 200
    assert L.moe_rows_cap(100, 8, 2, 1) == 200
    assert L.LIB.moe_rows_cap(-1, 8, 2, 0, 0) == -1
    # with token dropping no expert keeps more than `capacity` rows
    assert L.moe_rows_cap(100, 8, 2, 0, capacity=10) == 80
    assert L.moe_rows_cap(100, 8, 2, 16, capacity=10) == 80 + 8 * 15
    assert L.moe_rows_cap(100, 8, 2, 0, capacity=1000) == 200
    assert L.moe_rows_cap(32768, 64, 1, 128, capacity=512) == 32768 + 64 * 127
    assert L.moe_permute_workspace_bytes(4096, 64) >= 4 * 64 * 4
    assert L.LIB.moe_version() >= 200


def _ptr(v=16):
    return ctypes.c_void_p(v)


def test_validation_errors_need_no_gpu(L):
    lib = L.LIB
    # k > E
    st = lib.moe_route_topk(_ptr(), 8, 10, 8, 9, 0, 1, None, 0, 0, _ptr(), _ptr(), None)
    assert st == L.MOE_ERR_INVALID_ARG and "k=9" in L.last_error()
    # E above the router's limit
    st = lib.moe_route_topk(_ptr(), 300, 10, 300, 2, 0, 1, None, 0, 0, _ptr(), _ptr(), None)
    assert st == L.MOE_ERR_UNSUPPORTED
    # bad score function
    st = lib.moe_route_topk(_ptr(), 8, 10, 8, 2, 7, 1, None, 0, 0, _ptr(), _ptr(), None)
    assert st == L.MOE_ERR_INVALID_ARG
    # route: E not a multiple of num_groups; topk_group not dividing k
    st = lib.moe_route_topk(_ptr(), 10, 10, 10, 4, 0, 1, None, 4, 2, _ptr(), _ptr(), None)
    assert st == L.MOE_ERR_INVALID_ARG and "num_groups" in L.last_error()
    st = lib.moe_route_topk(_ptr(), 16, 10, 16, 4, 0, 1, None, 4, 3, _ptr(), _ptr(), None)
    assert st == L.MOE_ERR_INVALID_ARG and "topk_group" in L.last_error()
    # aux loss: workspace too small; bad score_fn in the backward
    st = lib.moe_aux_loss(_ptr(), 8, 1000, 8, 2, 0, _ptr(), 0.01, _ptr(), _ptr(), _ptr(), _ptr(),
                          4, None)
    assert st == L.MOE_ERR_INVALID_ARG and "workspace" in L.last_error()
    st = lib.moe_aux_loss_bwd(_ptr(), 8, 1000, 8, 2, 5, _ptr(), 0.01, 1.0, _ptr(), 8, 1, None)
    assert st == L.MOE_ERR_INVALID_ARG
    # fp8: bad format, column-wise copy too narrow, K not a multiple of 16
    st = lib.moe_fp8_quantize_act(_ptr(), 64, _ptr(), 4, 100, 64, 7, _ptr(), _ptr(), 64, _ptr(),
                                  1024, _ptr(), None)
    assert st == L.MOE_ERR_INVALID_ARG and "fmt" in L.last_error()
    st = lib.moe_fp8_quantize_act(_ptr(), 64, _ptr(), 4, 100, 64, 0, _ptr(), _ptr(), 64, _ptr(),
                                  128, _ptr(), None)
    assert st == L.MOE_ERR_INVALID_ARG and "leading dimension" in L.last_error()
    assert L.moe_fp8_padded_rows(100, 4) == 640 and L.moe_fp8_padded_rows(0, 1) == 128
    st = lib.moe_gmm_fp8(_ptr(), 64, 0, _ptr(), _ptr(), 24, 24 * 64, 0, _ptr(), _ptr(), 1, 100,
                         24, 64, 0, None, 0, _ptr(), 0, 64, None, 0, None, None, None)
    assert st == L.MOE_ERR_UNSUPPORTED
    st = lib.moe_tgmm_fp8(_ptr(), 64, 0, _ptr(), _ptr(), 1024, 1, _ptr(), _ptr(), 4, 100, 64, 64,
                          _ptr(), 0, 64, 64 * 64, 0, None, None)
    assert st == L.MOE_ERR_INVALID_ARG and "ldat" in L.last_error()
    # route backward: k > E, bad leading dimension
    st = lib.moe_route_topk_bwd(_ptr(), 8, _ptr(), _ptr(), _ptr(), 10, 8, 9, 0, 1, _ptr(), 8, None)
    assert st == L.MOE_ERR_INVALID_ARG
    st = lib.moe_route_topk_bwd(_ptr(), 8, _ptr(), _ptr(), _ptr(), 10, 8, 2, 0, 1, _ptr(), 4, None)
    assert st == L.MOE_ERR_INVALID_ARG
    # permute: rows_cap below the worst case
    st = lib.moe_permute(_ptr(), 64, _ptr(), 100, 64, 8, 2, 4, 0, _ptr(), 64, 100, _ptr(), _ptr(),
                         _ptr(), _ptr(), _ptr(), _ptr(), 1 << 20, None, None)
    assert st == L.MOE_ERR_INVALID_ARG and "rows_cap" in L.last_error()
    # permute: d not a multiple of 8
    st = lib.moe_permute(_ptr(), 64, _ptr(), 100, 60, 8, 2, 0, 0, _ptr(), 64, 200, _ptr(), _ptr(),
                         _ptr(), _ptr(), _ptr(), _ptr(), 1 << 20, None, None)
    assert st == L.MOE_ERR_UNSUPPORTED
    # permute: workspace too small
    st = lib.moe_permute(_ptr(), 64, _ptr(), 100, 64, 8, 2, 0, 0, _ptr(), 64, 200, _ptr(), _ptr(),
                         _ptr(), _ptr(), _ptr(), _ptr(), 4, None, None)
    assert st == L.MOE_ERR_INVALID_ARG and "workspace" in L.last_error()
    # gmm: N not a multiple of 8
    st = lib.moe_gmm(_ptr(), 64, _ptr(), 12, 64 * 12, 0, _ptr(), 1, 100, 64, 12, 0, None, 0, None,
                     0, None, 0, _ptr(), 0, 12, None, 0, None, 0, None, None)
    assert st == L.MOE_ERR_UNSUPPORTED
    # gmm: SWIGLU_FWD without C2
    st = lib.moe_gmm(_ptr(), 64, _ptr(), 64, 64 * 64, 0, _ptr(), 1, 100, 64, 64, 1, None, 0, None,
                     0, None, 0, _ptr(), 0, 64, None, 0, None, 0, None, None)
    assert st == L.MOE_ERR_INVALID_ARG
    # gmm: misaligned A
    st = lib.moe_gmm(_ptr(18), 64, _ptr(), 64, 64 * 64, 0, _ptr(), 1, 100, 64, 64, 0, None, 0,
                     None, 0, None, 0, _ptr(), 0, 64, None, 0, None, 0, None, None)
    assert st == L.MOE_ERR_UNSUPPORTED
    # gmm: in-place partial sum with bf16 C
    st = lib.moe_gmm(_ptr(), 64, _ptr(), 64, 64 * 64, 0, _ptr(), 1, 100, 64, 64, 0, None, 0,
                     _ptr(32), 64, None, 0, _ptr(32), 0, 64, None, 0, None, 0, None, None)
    assert st == L.MOE_ERR_INVALID_ARG
    # gmm: bias with a stride shorter than N
    st = lib.moe_gmm(_ptr(), 64, _ptr(), 64, 64 * 64, 0, _ptr(), 2, 100, 64, 64, 0, None, 0,
                     None, 0, _ptr(), 32, _ptr(), 0, 64, None, 0, None, 0, None, None)
    assert st == L.MOE_ERR_INVALID_ARG and "bias" in L.last_error()
    # gmm: bias with the SwiGLU backward
    st = lib.moe_gmm(_ptr(), 64, _ptr(), 64, 64 * 64, 1, _ptr(), 2, 100, 64, 64, 2, _ptr(), 128,
                     None, 0, _ptr(), 64, _ptr(), 0, 128, None, 0, None, 0, None, None)
    assert st == L.MOE_ERR_INVALID_ARG and "bias" in L.last_error()
    # gmm: a column-wise copy from the plain epilogue
    st = lib.moe_gmm(_ptr(), 64, _ptr(), 64, 64 * 64, 0, _ptr(), 1, 100, 64, 64, 0, None, 0,
                     None, 0, None, 0, _ptr(), 0, 64, None, 0, _ptr(), 256, None, None)
    assert st == L.MOE_ERR_INVALID_ARG and "Ct" in L.last_error()
    # gmm: a column-wise copy narrower than the padded group layout
    st = lib.moe_gmm(_ptr(), 64, _ptr(), 64, 64 * 64, 0, _ptr(), 2, 100, 64, 64, 1, None, 0,
                     None, 0, None, 0, _ptr(), 0, 64, _ptr(), 32, _ptr(), 128, None, None)
    assert st == L.MOE_ERR_INVALID_ARG and "ldct" in L.last_error()
    # group_colsum: N not a multiple of 8
    st = lib.moe_group_colsum(_ptr(), 64, _ptr(), 4, 100, 60, _ptr(), 64, None)
    assert st == L.MOE_ERR_UNSUPPORTED
    # group_colsum: null output
    st = lib.moe_group_colsum(_ptr(), 64, _ptr(), 4, 100, 64, None, 64, None)
    assert st == L.MOE_ERR_INVALID_ARG
    # tgmm: accumulate into bf16
    st = lib.moe_tgmm(_ptr(), 64, _ptr(), 64, _ptr(), 2, 100, 64, 64, _ptr(), 0, 64, 64 * 64, 1,
                      None, None)
    assert st == L.MOE_ERR_INVALID_ARG
    # combine: k above the limit
    st = lib.moe_combine(_ptr(), 64, _ptr(), _ptr(), 10, 17, 64, _ptr(), 64, None)
    assert st == L.MOE_ERR_UNSUPPORTED
    # unpermute_bwd: null dY
    st = lib.moe_unpermute_bwd(_ptr(), 64, _ptr(), 64, _ptr(), _ptr(), _ptr(), _ptr(), 10, 2, 64,
                               4, 20, None, 64, _ptr(), None)
    assert st == L.MOE_ERR_INVALID_ARG


def test_wait_limit_setting(L):
    default = L.moe_wait_limit_ns()
    assert default == 2_000_000_000
    assert L.LIB.moe_set_wait_limit_ns(10) == L.MOE_ERR_INVALID_ARG      # below 1 ms
    L.moe_set_wait_limit_ns(50_000_000)
    assert L.moe_wait_limit_ns() == 50_000_000
    L.moe_set_wait_limit_ns(default)
    assert L.moe_wait_limit_ns() == default


def test_product_path_never_touches_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in src.replace("the oracle", ""), fn
                assert "moe_ref" not in src, fn


def test_layer_rejects_uneven_chunks(L):
    """K-chunks must tile d_model: a remainder would leave columns of x and wi
    out of the up-projection (checked before any device memory is touched)."""
    from mixture_experts_grouped_router_gb300 import layer
    with pytest.raises(ValueError, match="does not divide"):
        layer.MoEBuffers(layer.LayerShape(T=8, d=264, f=64, E=2, k=1, num_chunks=16),
                         device="cpu")
