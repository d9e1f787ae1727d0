"""The C-ABI library on the CPU: it builds, loads, exports every function that
include/tim.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tim.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from rollout_logprob_consistency_gb300 import binding
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(tim_[a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("tim_logprob", "tim_logprob_workspace_size", "tim_compare",
                 "tim_compare_workspace_size", "tim_status_sync", "tim_status_string",
                 "tim_workspace_init", "tim_rmsnorm_rows", "tim_lmhead_lse", "tim_lse_finalize",
                 "tim_abi_version"):
        assert must in names


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libtim.so does not export {name}"
    assert lib.tim_abi_version() == 1


def test_status_strings(lib):
    from rollout_logprob_consistency_gb300 import binding
    for code, name in binding.STATUS_NAMES.items():
        assert binding.status_string(code) == name
    assert binding.status_string(99) == "TIM_ERR_UNKNOWN"


def test_workspace_sizes(lib):
    from rollout_logprob_consistency_gb300 import binding
    assert binding.logprob_workspace_size(0, 64, 10) == 0
    assert binding.logprob_workspace_size(1, 100, 10) == 0   # d not a multiple of 64
    T, d, V = 32768, 4096, 151936
    n_tiles = (V + 255) // 256
    need = T * d * 2 + (T // 32) * n_tiles * 32 * 16 + T * 4
    got = binding.logprob_workspace_size(T, d, V)
    assert need <= got <= need + 4 * 1024
    assert binding.compare_workspace_size(10, 1) >= 256


def test_argument_errors_need_no_gpu(lib):
    from rollout_logprob_consistency_gb300.binding import STATUS
    fake = 1 << 20   # never dereferenced: validation fails first
    ws = 1 << 24
    # null pointer
    assert lib.tim_logprob(None, fake, fake, fake, 4, 64, 10, 1.0, 0.0, fake, fake, fake,
                           ws, 1 << 30, None) == STATUS["TIM_ERR_INVALID_ARG"]
    # d not a multiple of 64
    assert lib.tim_logprob(fake, fake, fake, fake, 4, 96, 10, 1.0, 0.0, fake, fake, fake,
                           ws, 1 << 30, None) == STATUS["TIM_ERR_SHAPE"]
    # T < 1
    assert lib.tim_logprob(fake, fake, fake, fake, 0, 64, 10, 1.0, 0.0, fake, fake, fake,
                           ws, 1 << 30, None) == STATUS["TIM_ERR_SHAPE"]
    # temperature <= 0, NaN eps
    assert lib.tim_logprob(fake, fake, fake, fake, 4, 64, 10, 0.0, 0.0, fake, fake, fake,
                           ws, 1 << 30, None) == STATUS["TIM_ERR_INVALID_ARG"]
    assert lib.tim_logprob(fake, fake, fake, fake, 4, 64, 10, 1.0, float("nan"), fake, fake,
                           fake, ws, 1 << 30, None) == STATUS["TIM_ERR_INVALID_ARG"]
    # misaligned hidden
    assert lib.tim_logprob(fake + 2, fake, fake, fake, 4, 64, 10, 1.0, 0.0, fake, fake, fake,
                           ws, 1 << 30, None) == STATUS["TIM_ERR_INVALID_ARG"]
    # workspace too small / misaligned
    assert lib.tim_logprob(fake, fake, fake, fake, 4, 64, 10, 1.0, 0.0, fake, fake, fake,
                           ws, 100, None) == STATUS["TIM_ERR_WORKSPACE"]
    assert lib.tim_logprob(fake, fake, fake, fake, 4, 64, 10, 1.0, 0.0, fake, fake, fake,
                           ws + 16, 1 << 30, None) == STATUS["TIM_ERR_WORKSPACE"]
    # compare: bad cap, bad sizes, null
    assert lib.tim_compare(fake, fake, fake, fake, 1, fake, 8, 0.0, fake, None, ws, 4096,
                           None) == STATUS["TIM_ERR_INVALID_ARG"]
    assert lib.tim_compare(fake, fake, fake, fake, 0, fake, 8, 2.0, fake, None, ws, 4096,
                           None) == STATUS["TIM_ERR_SHAPE"]
    assert lib.tim_compare(fake, None, fake, fake, 1, fake, 8, 2.0, fake, None, ws, 4096,
                           None) == STATUS["TIM_ERR_INVALID_ARG"]
    # more than 2^31 - 1 tokens: rejected (per-sequence token counts are 32-bit inside)
    big = 1 << 31
    assert lib.tim_compare(fake, fake, fake, fake, 1, fake, big, 2.0, fake, None, ws, 1 << 62,
                           None) == STATUS["TIM_ERR_SHAPE"]
    assert lib.tim_compare_diag(fake, fake, fake, None, None, None, fake, 1, fake, big, 2.0, 0.5,
                                2.0, fake, ws, 1 << 62, None) == STATUS["TIM_ERR_SHAPE"]
    assert lib.tim_workspace_init(None, 0, None) == STATUS["TIM_ERR_WORKSPACE"]


def test_variant_sizes_and_argument_errors_need_no_gpu(lib):
    """The next-row entry points validate before touching the device."""
    from rollout_logprob_consistency_gb300.binding import STATUS
    fake, ws = 1 << 20, 1 << 24
    inv, shape = STATUS["TIM_ERR_INVALID_ARG"], STATUS["TIM_ERR_SHAPE"]
    # workspace sizes: zero for invalid shapes, covering the parts for valid ones
    assert lib.tim_logprob_fp8_workspace_size(4, 192, 10) == 0          # d % 128
    assert lib.tim_logprob_fp8_workspace_size(4, 256, 10) > lib.tim_logprob_workspace_size(4, 256, 10)
    assert lib.tim_logprob_fp32_workspace_size(4, 96, 10) == 0
    assert lib.tim_logprob_fp32_workspace_size(128, 64, 10) >= 2 * 128 * 64 * 4
    T, d, V = 1000, 256, 3000
    Tp, Vp = 1024, 3008
    # y bf16 [Tp][d] and G bf16 [Tp][Vp]; the products read G, W and y in place
    assert lib.tim_logprob_backward_workspace_size(T, d, V) >= 2 * Tp * Vp + 2 * Tp * d
    assert lib.tim_logprob_backward_workspace_size(T, d, V) < 3 * Tp * Vp
    assert lib.tim_rmsnorm_backward_workspace_size(T, d) >= 4 * T + 4 * d * 4
    assert lib.tim_rmsnorm_backward_workspace_size(T, 100) == 0
    assert lib.tim_selftest_workspace_size() > 0
    assert lib.tim_compare_diag_workspace_size(0, 1) == 0
    # FP8: d not a multiple of 128; null scales
    assert lib.tim_logprob_fp8(fake, fake, fake, fake, fake, 4, 192, 300, 1.0, 0.0, fake, fake,
                               fake, ws, 1 << 30, None) == shape
    assert lib.tim_logprob_fp8(fake, fake, fake, None, fake, 4, 256, 300, 1.0, 0.0, fake, fake,
                               fake, ws, 1 << 30, None) == inv
    assert lib.tim_quantize_fp8_rows(fake, 4, 24, fake, fake, None) == shape   # K % 16
    # FP32 / split: misaligned W part, n not a multiple of 4
    assert lib.tim_logprob_fp32(fake, fake, fake + 4, fake, fake, 4, 64, 300, 1.0, 0.0, fake,
                                fake, fake, ws, 1 << 30, None) == inv
    assert lib.tim_split_tf32(fake, 6, fake, fake, None) == shape
    # backward: accumulate flag, temperature, misaligned outputs
    assert lib.tim_logprob_backward(fake, fake, fake, fake, fake, fake, 4, 64, 300, 1.0, 0.0,
                                    fake, fake, 2, ws, 1 << 30, None) == inv
    assert lib.tim_logprob_backward(fake, fake, fake, fake, fake, fake, 4, 64, 300, -1.0, 0.0,
                                    fake, fake, 0, ws, 1 << 30, None) == inv
    assert lib.tim_logprob_backward(fake, fake, fake, fake, fake, fake, 4, 64, 300, 1.0, 0.0,
                                    fake + 4, fake, 0, ws, 1 << 30, None) == inv
    assert lib.tim_rmsnorm_backward(fake, fake, fake, 4, 96, 0.0, fake, fake, 0, ws, 1 << 30,
                                    None) == shape
    assert lib.tim_rmsnorm_backward(fake, fake, fake, 4, 64, -1.0, fake, fake, 0, ws, 1 << 30,
                                    None) == inv
    # processed head: exactly one head output given
    assert lib.tim_processed_logprob_head(fake, fake, fake, fake, 4, 64, 5000, 1.0, 0.0, 4, 1.0,
                                          fake, fake, fake, fake, None, ws, 1 << 30,
                                          None) == inv
    # self-test limit out of range
    assert lib.tim_selftest_wait_timeout(0, ws, 1 << 30, None) == inv
    assert lib.tim_selftest_wait_timeout(2001, ws, 1 << 30, None) == inv


def test_product_path_does_not_import_oracle():
    """The package and its binding never import the oracle (test infrastructure only)."""
    pkg = os.path.join(ROOT, "rollout_logprob_consistency_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", txt, flags=re.M), f
                assert "oracle/" not in txt, f
