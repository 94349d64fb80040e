"""C ABI checks that need no GPU: the library builds, loads, exports every
symbol include/bimoe.h declares, and rejects bad arguments on the host."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from invariant_moe_gb300 import _build
    _build.build()
    import invariant_moe_gb300 as bm
    return bm.load_library()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "bimoe.h")).read()
    return sorted(set(re.findall(r"BI_API\s+[\w\s\*]+?\b(bi_\w+)\s*\(", src)))


def test_header_and_binding_agree():
    import invariant_moe_gb300 as bm
    assert declared_symbols() == sorted(bm.EXPORTS)


def test_status_and_device_error_codes_agree():
    """The binding's names for the status and device error codes are the
    header's values."""
    import invariant_moe_gb300 as bm
    src = open(os.path.join(ROOT, "include", "bimoe.h")).read()
    deverr = {int(v): n for n, v in re.findall(r"#define\s+BI_DEVERR_(\w+)\s+(\d+)", src)}
    assert sorted(deverr) == sorted(bm.DEVERR)
    assert deverr[0] == "NONE" and deverr[3] == "WAIT_TIMEOUT" and deverr[4] == "BAD_PERMUTATION"


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert lib.bi_status_str(0) == b"BI_OK"
    assert lib.bi_status_str(3) == b"BI_ERR_WORKSPACE"
    assert lib.bi_version().startswith(b"bimoe")


def test_workspace_sizes(lib):
    qwen = lib.bi_moe_workspace_bytes(4096, 2048, 128, 8, 768)
    assert qwen % 256 == 0
    P = 4096 * 8
    # gathered rows + activations + fp32 contributions dominate
    assert qwen >= P * (2048 * 2 + 768 * 2 + 2048 * 4)
    assert lib.bi_moe_workspace_bytes(4096, 2000, 128, 8, 768) == 0   # H % 128 != 0
    assert lib.bi_moe_workspace_bytes(16, 2048, 8, 9, 768) == 0       # top_k > E
    assert lib.bi_moe_workspace_bytes(0, 2048, 128, 8, 768) > 0


def test_router_topk_host_checks(lib):
    """The router + top-k call checks its arguments on the host."""
    nul = ctypes.c_void_p(None)
    fake = ctypes.c_void_p(0x10000)
    args = lambda N, k, ids: (fake, fake, nul, fake, nul, ids, fake, 4096, 4096, N, k, nul)
    assert lib.bi_router_topk(*args(600, 8, fake)) == 2          # N > 512
    assert lib.bi_router_topk(*args(256, 17, fake)) == 1         # top_k > 16
    assert lib.bi_router_topk(*args(256, 8, nul)) == 1           # no ids buffer
    assert lib.bi_router_topk(fake, fake, nul, fake, nul, fake, fake, 4, 100, 256, 8, nul) == 2  # K % 128
    # M == 0 is a no-op
    assert lib.bi_router_topk(nul, nul, nul, nul, nul, nul, nul, 0, 4096, 256, 8, nul) == 0


def test_router_bf16_host_checks(lib):
    nul = ctypes.c_void_p(None)
    fake = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)   # 8-byte but not 16-byte aligned
    assert lib.bi_router_gemm_bf16(fake, fake, nul, fake, 4, 100, 256, nul) == 2   # K % 128
    assert lib.bi_router_gemm_bf16(odd, fake, nul, fake, 4, 128, 256, nul) == 1    # misaligned x
    assert lib.bi_router_gemm_bf16_schedule(fake, fake, nul, fake, 4, 128, 256, 10, nul) == 1
    # the cluster-split schedules need K/128 to split into 2..8 CTAs of 4 or 8 slices
    assert lib.bi_router_gemm_bf16_schedule(fake, fake, nul, fake, 4, 512, 256, 4, nul) == 2
    assert lib.bi_router_gemm_schedule(fake, fake, nul, fake, 4, 36 * 128, 256, 8, nul) == 2
    assert lib.bi_router_topk_bf16(fake, fake, nul, fake, nul, fake, fake, 4, 128, 600, 8, nul) == 2
    assert lib.bi_router_gemm_bf16(nul, nul, nul, nul, 0, 128, 256, nul) == 0      # M == 0


def test_topk_window_host_checks(lib):
    nul = ctypes.c_void_p(None)
    fake = ctypes.c_void_p(0x10000)
    assert lib.bi_topk_window(fake, 9000, nul, nul, 4, 9000, 512, fake, nul) == 2   # > 8192 columns
    assert lib.bi_topk_window(fake, 100, nul, nul, 4, 200, 512, fake, nul) == 1     # ld < num_cols
    assert lib.bi_topk_window(fake, 8192, nul, nul, 4, 8192, 0, fake, nul) == 1     # k < 1
    assert lib.bi_topk_window(fake, 8192, nul, nul, 4, 8192, 512, nul, nul) == 1    # no output
    assert lib.bi_topk_window(nul, 8192, nul, nul, 0, 8192, 512, nul, nul) == 0     # no rows


def test_gemm_variant_setting(lib):
    """The expert-GEMM variant is a host-side setting: no GPU needed."""
    prev = ctypes.c_int32(-1)
    assert lib.bi_moe_gemm_variant(5, None) == 1
    assert lib.bi_moe_gemm_variant(-1, None) == 1
    assert lib.bi_moe_gemm_variant(1, ctypes.byref(prev)) == 0 and prev.value == 0
    assert lib.bi_moe_gemm_variant(0, ctypes.byref(prev)) == 0 and prev.value == 1


def test_decode_fused_setting_and_probe_arguments(lib):
    """The decode layer's one- or two-launch setting is host-side, and the
    bounded-wait probe rejects an unknown wait kind before any launch."""
    prev = ctypes.c_int32(-1)
    assert lib.bi_moe_decode_fused(2, None) == 1
    assert lib.bi_moe_decode_fused(-1, None) == 1
    assert lib.bi_moe_decode_fused(1, ctypes.byref(prev)) == 0 and prev.value == 0
    assert lib.bi_moe_decode_fused(0, ctypes.byref(prev)) == 0 and prev.value == 1
    assert lib.bi_wait_timeout_probe(2, ctypes.c_void_p(None)) == 1
    assert lib.bi_wait_timeout_probe(-1, ctypes.c_void_p(None)) == 1


def test_host_side_rejections(lib):
    """Argument checks run on the host and never touch the GPU."""
    nul = ctypes.c_void_p(None)
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: rejected first
    odd = ctypes.c_void_p(0x10004)         # not 16-byte aligned
    # K not a multiple of 128
    assert lib.bi_router_gemm(fake, fake, nul, fake, 4, 100, 256, nul) == 2
    # misaligned x
    assert lib.bi_router_gemm(odd, fake, nul, fake, 4, 128, 256, nul) == 1
    # null x with M > 0
    assert lib.bi_router_gemm(nul, fake, nul, fake, 4, 128, 256, nul) == 1
    assert b"null" in lib.bi_last_error_message()
    # M == 0 is a no-op
    assert lib.bi_router_gemm(nul, nul, nul, nul, 0, 128, 256, nul) == 0
    # top_k > E, E too large
    assert lib.bi_topk(fake, nul, fake, fake, 4, 8, 9, nul) == 1
    assert lib.bi_topk(fake, nul, fake, fake, 4, 600, 8, nul) == 2
    # null ids with M > 0 (probs may be NULL, ids and wts may not)
    assert lib.bi_topk(fake, fake, nul, fake, 4, 256, 8, nul) == 1
    # MoE: workspace too small, unsupported H
    assert lib.bi_moe_forward(fake, fake, fake, fake, fake, fake, 4, 2048, 128, 8, 768,
                              fake, 1024, nul) == 3
    assert lib.bi_moe_forward(fake, fake, fake, fake, fake, fake, 4, 2000, 128, 8, 768,
                              fake, 1 << 30, nul) == 2
    assert lib.bi_moe_forward(nul, nul, nul, nul, nul, nul, 0, 2048, 128, 8, 768,
                              nul, 0, nul) == 0
    assert lib.bi_moe_combine(fake, fake, 4, 2046, 8, nul) == 1
    assert lib.bi_moe_combine_consume(fake, fake, 4, 2046, 8, nul) == 1
    assert lib.bi_moe_combine_consume(fake, fake, 4, 2048, 17, nul) == 1
    assert lib.bi_moe_combine_consume(nul, nul, 0, 2048, 8, nul) == 0


def test_moe_wrappers_check_shapes_first():
    """The layer wrappers reject mismatched weight or routing shapes before
    any pointer reaches the library (no GPU needed)."""
    import torch
    import invariant_moe_gb300 as bm
    M, H, E, I, k = 4, 256, 8, 128, 2
    x = torch.zeros(M, H, dtype=torch.bfloat16)
    ids = torch.zeros(M, k, dtype=torch.int32)
    wts = torch.zeros(M, k)
    w13 = torch.zeros(E, 2 * I, H, dtype=torch.bfloat16)
    w2 = torch.zeros(E, H, I, dtype=torch.bfloat16)
    for fn in (bm.bi_moe_forward, bm.bi_moe_forward_noalloc):
        with pytest.raises(ValueError, match="w13"):
            fn(x, ids, wts, w13, torch.zeros(E, H, I + 128, dtype=torch.bfloat16))
        with pytest.raises(ValueError, match="w13"):
            fn(x, ids, wts, torch.zeros(E, 2 * I, H + 128, dtype=torch.bfloat16), w2)
        with pytest.raises(ValueError, match="ids"):
            fn(x, ids, torch.zeros(M, k + 1), w13, w2)
        with pytest.raises(ValueError, match="ids"):
            fn(x, ids[:2], wts[:2], w13, w2)


def test_binding_rejects_cpu_tensors():
    import torch
    import invariant_moe_gb300 as bm
    with pytest.raises(ValueError):
        bm.bi_router_gemm(torch.zeros(2, 128), torch.zeros(4, 128))
