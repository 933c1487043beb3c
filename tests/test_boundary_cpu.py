"""The C-ABI library without a GPU: it loads, exports every function the
header declares, and rejects bad arguments on the host before touching CUDA."""

import os
import re

import pytest

import flashattention_fa_fwd_gb300 as fa
from flashattention_fa_fwd_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_binding.library_path()):
        from flashattention_fa_fwd_gb300.build import build

        build()
    return fa.load_library()


def test_exports_every_declared_function(lib):
    declared = _declared_functions()
    assert set(_binding.EXPORTED) <= set(declared), declared
    for name in declared:
        assert hasattr(lib, name), f"libfa_fwd.so does not export {name}"


def test_status_strings(lib):
    assert [fa.fa_status_string(i) for i in range(5)] == [
        "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT"]
    assert fa.fa_status_string(99) == "FA_ERR_UNKNOWN"


A = 1 << 24   # fake, 16-byte aligned, non-overlapping device addresses (never dereferenced)
PTRS = (A, 2 * A, 3 * A, 4 * A, 5 * A)


@pytest.mark.parametrize("raw", [fa.fa_fwd_raw, fa.fa_fwd_f32_raw])
@pytest.mark.parametrize("args,want", [
    (dict(B=-1), fa.FA_ERR_INVALID_ARG),
    (dict(N=-5), fa.FA_ERR_INVALID_ARG),
    (dict(D=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.5), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(o=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(k=0), fa.FA_ERR_INVALID_ARG),
    (dict(q=A + 8), fa.FA_ERR_INVALID_ARG),
    (dict(lse=5 * A + 2), fa.FA_ERR_INVALID_ARG),
    (dict(o=A + 16), fa.FA_ERR_INVALID_ARG),          # o overlaps q
    (dict(lse=4 * A + 64), fa.FA_ERR_INVALID_ARG),    # lse inside o
    (dict(M=1 << 31), fa.FA_ERR_INVALID_ARG),
    (dict(D=300), fa.FA_ERR_UNSUPPORTED),
    (dict(B=0), fa.FA_OK),                             # empty problem: nothing launched
    (dict(M=0), fa.FA_OK),
    (dict(H=0, q=0, o=0, lse=0), fa.FA_OK),
])
def test_host_validation(lib, raw, args, want):
    a = dict(zip(("q", "k", "v", "o", "lse"), PTRS), B=1, H=2, M=256, N=512, D=64, scale=0.125)
    a.update(args)
    st = raw(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["M"], a["N"], a["D"], a["scale"], False, 0)
    assert st == want, (st, fa.fa_last_error())
    if want != fa.FA_OK:
        assert fa.fa_last_error()


@pytest.mark.parametrize("D", [32, 80, 100, 192, 256])
def test_bf16_head_dims_outside_the_kernel_set(lib, D):
    st = fa.fa_fwd_raw(*PTRS, 1, 1, 128, 128, D, 0.1, True, 0)
    assert st == fa.FA_ERR_UNSUPPORTED


def test_empty_keys_need_no_key_pointers(lib):
    # N == 0 with null k and v passes validation; with B == 0 nothing launches.
    assert fa.fa_fwd_raw(A, 0, 0, 4 * A, 5 * A, 0, 1, 128, 0, 64, 0.1, False, 0) == fa.FA_OK


def test_binding_rejects_bad_tensors_without_gpu(lib):
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, q.clone(), torch.zeros(8), 0.125)       # CPU tensors
    with pytest.raises(TypeError):
        fa.fa_fwd(q.float(), q, q, q.clone(), torch.zeros(8), 0.125)


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "_LIB_PATH", "/nonexistent/libfa_fwd.so")
    with pytest.raises(RuntimeError, match="not built"):
        _binding.load_library()


def test_splitkv_workspace_size_and_checks(lib):
    # num_splits * B*H*M * (D + 1) * 4
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 8, 1000, 96, 3) == 3 * 16 * 1000 * 97 * 4
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 8, 1000, 96, 1) == 0
    assert fa.fa_fwd_splitkv_workspace_bytes(2, 8, 1000, 96, 0) == -1
    need = fa.fa_fwd_splitkv_workspace_bytes(1, 2, 256, 64, 2)
    W = 64 * A
    args = (*PTRS, 1, 2, 256, 512, 64, 0.125, False)
    assert fa.fa_fwd_splitkv_raw(*args, 2, W, need - 4, 0) == fa.FA_ERR_INVALID_ARG     # too small
    assert fa.fa_fwd_splitkv_raw(*args, 2, 0, need, 0) == fa.FA_ERR_INVALID_ARG          # missing
    assert fa.fa_fwd_splitkv_raw(*args, 2, W + 4, need, 0) == fa.FA_ERR_INVALID_ARG      # misaligned
    assert fa.fa_fwd_splitkv_raw(*args, 2, A, need, 0) == fa.FA_ERR_INVALID_ARG          # overlaps q
    assert fa.fa_fwd_splitkv_raw(*args, 17, W, need, 0) == fa.FA_ERR_INVALID_ARG         # too many splits
    assert fa.fa_fwd_splitkv_raw(A, 2 * A, 3 * A, 4 * A, 5 * A, 0, 2, 256, 512, 64, 0.125, False,
                                 2, W, need, 0) == fa.FA_OK                                # empty problem


def test_host_entry_workspace_size_and_checks(lib):
    # two slots; per slot q, k, v, o (bf16) and lse (fp32), each padded to 256 bytes
    def pad(x):
        return (x + 255) // 256 * 256
    hc, M, N, D = 3, 100, 300, 64
    slot = pad(hc * M * D * 2) + 2 * pad(hc * N * D * 2) + pad(hc * M * D * 2) + pad(hc * M * 4)
    assert fa.fa_fwd_host_workspace_bytes(2, 4, M, N, D, hc) == 2 * slot
    # default chunk: up to eight chunks, none with less than 32 MiB of q, k, v; never more heads than exist
    assert fa.fa_fwd_host_workspace_bytes(8, 32, M, N, D, 0) == fa.fa_fwd_host_workspace_bytes(8, 32, M, N, D, 256)
    assert (fa.fa_fwd_host_workspace_bytes(8, 32, 4096, 4096, 128, 0)
            == fa.fa_fwd_host_workspace_bytes(8, 32, 4096, 4096, 128, 32))   # 805 MB in: eight chunks
    assert (fa.fa_fwd_host_workspace_bytes(2, 8, 1000, 3000, 96, 0)
            == fa.fa_fwd_host_workspace_bytes(2, 8, 1000, 3000, 96, 16))     # 21 MB in: one chunk
    assert fa.fa_fwd_host_workspace_bytes(1, 2, M, N, D, 50) == fa.fa_fwd_host_workspace_bytes(1, 2, M, N, D, 2)
    assert fa.fa_fwd_host_workspace_bytes(0, 2, M, N, D, 0) == 0
    assert fa.fa_fwd_host_workspace_bytes(1, 2, M, N, D, -1) == -1
    need = fa.fa_fwd_host_workspace_bytes(1, 2, 256, 512, 64, 0)
    W = 64 * A
    args = (*PTRS, 1, 2, 256, 512, 64, 0.125, False)
    assert fa.fa_fwd_host_raw(*args, 0, W, need - 256, 0) == fa.FA_ERR_INVALID_ARG   # too small
    assert fa.fa_fwd_host_raw(*args, 0, 0, need, 0) == fa.FA_ERR_INVALID_ARG          # missing
    assert fa.fa_fwd_host_raw(*args, 0, W + 16, need, 0) == fa.FA_ERR_INVALID_ARG     # not 256-aligned
    assert fa.fa_fwd_host_raw(*args, -1, W, need, 0) == fa.FA_ERR_INVALID_ARG         # negative chunk
    assert fa.fa_fwd_host_raw(*PTRS, 1, 2, 256, 512, 48, 0.125, False, 0, W, need, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_host_raw(*PTRS, 0, 2, 256, 512, 64, 0.125, False, 0, W, need, 0) == fa.FA_OK  # empty


def test_wait_selftest_rejects_bad_limits(lib):
    assert fa.fa_selftest_wait_timeout(0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_selftest_wait_timeout(2_000_000) == fa.FA_ERR_INVALID_ARG


def test_bwd_workspace_size_and_checks(lib):
    assert fa.fa_bwd_workspace_bytes(2, 3, 100) == 2 * 2 * 3 * 128 * 4   # Dl and base-2 LSE, rows padded to 128
    assert fa.fa_bwd_workspace_bytes(-1, 3, 100) == -1
    W = 64 * A
    grads = (6 * A, 7 * A, 8 * A)
    args = (*PTRS, 9 * A, *grads, 1, 2, 256, 512, 64, 0.125, False)
    need = fa.fa_bwd_workspace_bytes(1, 2, 256)
    assert fa.fa_bwd_raw(*args, 0, need, 0) == fa.FA_ERR_INVALID_ARG             # missing workspace
    assert fa.fa_bwd_raw(*args, W, need - 4, 0) == fa.FA_ERR_INVALID_ARG         # short workspace
    assert fa.fa_bwd_raw(*PTRS, 9 * A, 0, 7 * A, 8 * A, 1, 2, 256, 512, 64, 0.125, False, W, need, 0) \
        == fa.FA_ERR_INVALID_ARG                                                  # null dq
    assert fa.fa_bwd_raw(*PTRS, 9 * A, 6 * A + 4, 7 * A, 8 * A, 1, 2, 256, 512, 64, 0.125, False, W, need, 0) \
        == fa.FA_ERR_INVALID_ARG                                                  # misaligned dq
    assert fa.fa_bwd_raw(*PTRS, 9 * A, *grads, 1, 2, 256, 512, 192, 0.125, False, W, need, 0) \
        == fa.FA_ERR_UNSUPPORTED                                                  # D > 128
    assert fa.fa_bwd_raw(*PTRS, 9 * A, 6 * A, 6 * A, 8 * A, 1, 2, 256, 512, 64, 0.125, False, W, need, 0) \
        == fa.FA_ERR_INVALID_ARG                                                  # dq overlaps dk
    assert fa.fa_bwd_raw(*PTRS, 9 * A, *grads, 0, 2, 256, 512, 64, 0.125, False, 0, 0, 0) == fa.FA_OK  # empty


def test_f32x3_workspace_size_and_checks(lib):
    # 16 bytes per (head, key, column), keys padded to the key block (64 for D >= 96, 32 below).
    assert fa.fa_fwd_f32x3_workspace_bytes(2, 3, 100, 64) == 2 * 3 * 128 * 64 * 16
    assert fa.fa_fwd_f32x3_workspace_bytes(1, 1, 33, 64) == 64 * 64 * 16
    assert fa.fa_fwd_f32x3_workspace_bytes(1, 1, 33, 128) == 64 * 128 * 16
    assert fa.fa_fwd_f32x3_workspace_bytes(1, 1, 65, 128) == 128 * 128 * 16
    assert fa.fa_fwd_f32x3_workspace_bytes(1, 1, 0, 64) == 0
    assert fa.fa_fwd_f32x3_workspace_bytes(-1, 1, 1, 64) == -1
    W = 64 * A
    need = fa.fa_fwd_f32x3_workspace_bytes(1, 2, 512, 64)
    args = (*PTRS, 1, 2, 256, 512, 64, 0.125, False)
    assert fa.fa_fwd_f32x3_raw(*args, 0, need, 0) == fa.FA_ERR_INVALID_ARG          # missing workspace
    assert fa.fa_fwd_f32x3_raw(*args, W, need - 16, 0) == fa.FA_ERR_INVALID_ARG     # short workspace
    assert fa.fa_fwd_f32x3_raw(*args, W + 16, need, 0) == fa.FA_ERR_INVALID_ARG     # misaligned workspace
    assert fa.fa_fwd_f32x3_raw(*args, A, need, 0) == fa.FA_ERR_INVALID_ARG          # overlaps q
    for D in (8, 48, 80, 112, 256):
        assert fa.fa_fwd_f32x3_raw(*PTRS, 1, 2, 256, 512, D, 0.125, False, W, 1 << 30, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_f32x3_raw(*PTRS, 1, 2, 256, 512, 64, float("nan"), False, W, need, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_f32x3_raw(*PTRS, 0, 2, 256, 512, 64, 0.125, False, 0, 0, 0) == fa.FA_OK  # empty
