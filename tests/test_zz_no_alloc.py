"""The allocation-free decode entry point, called through the C ABI.

sink_attn_decode_static_workspace serves callers that cannot allocate device memory
(a plugin handed only its input and output buffers by a framework that owns every
allocation, or a decode loop that must not call cudaMalloc because it can synchronise
the device): its split-KV scratch is a fixed array inside the library. This file is
collected last on purpose, so a run that stops at its first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import gqa_attention_head_gb300 as sa
import oracle
from gqa_attention_head_gb300 import _build
from gqa_attention_head_gb300 import workloads as wl
from parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    _build.build()
    lib = sa.load_library()
    p, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.sink_attn_decode_static_workspace.argtypes = [
        p, p, p, i32, i32, p, i32, p, i32, i32, i32, i32, i32, p, i32, ctypes.c_float, i32, p, p]
    lib.sink_attn_decode_static_workspace.restype = ctypes.c_int
    return lib


def ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_static(lib, dc, q, kc, vc, pt, sl, sk, out, max_seq_len, kv_chunk, window=0):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sink_attn_decode_static_workspace(
        ptr(q), ptr(kc), ptr(vc), kc.shape[0], kc.shape[2], ptr(pt), pt.shape[1], ptr(sl),
        q.shape[0], max_seq_len, q.shape[1], kc.shape[1], q.shape[2], ptr(sk), window,
        dc.scale, kv_chunk, ptr(out), stream)


@pytest.mark.parametrize("window", [0, 1500])
def test_static_workspace_matches_caller_workspace_twice(lib, window):
    # 16 sequences of up to 5000 positions with 512-token chunks: up to 10 chunks each
    # (3 with the 1500-token window), 16*64*10*65*4 bytes of scratch (2.7 MB), well inside
    # the 16 MiB array. Every case has sequences that span several chunks, so the partial
    # results do pass through the array.
    dc = wl.decode_case([5000, 1, 17, 1024, 1025, 4096, 3000, 0, 2222, 4999, 512, 513, 77,
                         4000, 2500, 1500], 64, 8, 64, seed=31, kv_chunk=512)
    q, kc, vc = dc.q.cuda(), dc.k_cache.cuda(), dc.v_cache.cuda()
    pt, sl, sk = dc.page_table.cuda(), dc.seq_lens.cuda(), dc.sinks.cuda()
    ref = sa.sink_attn_decode(q, kc, vc, pt, sl, sk, dc.max_seq_len, window=window,
                              scale=dc.scale, kv_chunk=512)
    torch.cuda.synchronize()
    exact = oracle.decode(wl.bf16_bits(dc.q), wl.bf16_bits(dc.k_cache), wl.bf16_bits(dc.v_cache),
                          dc.page_table.numpy(), dc.seq_lens.numpy(), dc.sinks.numpy(),
                          window=window, scale=dc.scale)
    for call in range(2):  # the second call reuses the array the first one left behind
        out = torch.full_like(q, float("nan"))
        st = call_static(lib, dc, q, kc, vc, pt, sl, sk, out, dc.max_seq_len, 512, window)
        assert st == 0, sa.sink_attn_status_string(st)
        torch.cuda.synchronize()
        assert_parity(out, exact, f"static scratch vs oracle, call {call + 1}", strict=True)
        assert_parity(out, ref.double().cpu().numpy(), f"static scratch vs caller scratch, "
                      f"call {call + 1}", strict=True)
    st, bits = sa.sink_attn_read_device_error()
    assert st == 0, f"device error word {bits:#x}"


def test_static_workspace_rejects_sizes_beyond_its_limit(lib):
    # 64 sequences x 64 heads x 32 chunks x (128 + 1) floats = 67 MB > 16 MiB.
    B, hq, hkv, d = 64, 64, 8, 128
    q = torch.zeros((B, hq, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, hkv, 16, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    pt = torch.zeros((B, 512), dtype=torch.int32, device="cuda")
    sl = torch.zeros((B,), dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 2.0)
    dc = wl.DecodeCase(q, kc, vc, pt, sl, None, 0, d ** -0.5)
    assert sa.sink_attn_decode_workspace_bytes(B, hq, d, 8192, 256) > (16 << 20)
    st = call_static(lib, dc, q, kc, vc, pt, sl, None, out, 8192, 256)
    assert st == 3  # SINK_ATTN_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.all(out == 2.0)
