"""GPU parity of sink_attn_decode (split-KV kernel + merge, called through the C ABI)
against the fp64 oracle, element by element, on seeded paged inputs; plus edge cases,
guard bands and the device-side checks."""
import numpy as np
import pytest
import torch

import gqa_attention_head_gb300 as sa
import oracle
from gqa_attention_head_gb300 import workloads as wl
from parity import assert_parity

pytestmark = pytest.mark.gpu

bits = wl.bf16_bits


@pytest.fixture(scope="module", autouse=True)
def _library():
    from gqa_attention_head_gb300 import _build
    _build.build()
    sa.load_library()
    sa.sink_attn_read_device_error()
    yield


def gpu_decode(dc, window=None, kv_chunk=None, out=None, workspace=None, max_seq_len=None,
               k_cache=None, v_cache=None, page_table=None):
    kc = dc.k_cache if k_cache is None else k_cache
    vc = dc.v_cache if v_cache is None else v_cache
    return sa.sink_attn_decode(
        dc.q.cuda(), kc.cuda(), vc.cuda(), (dc.page_table if page_table is None else page_table).cuda(),
        dc.seq_lens.cuda(), None if dc.sinks is None else dc.sinks.cuda(),
        dc.max_seq_len if max_seq_len is None else max_seq_len,
        window=dc.window if window is None else window, scale=dc.scale,
        kv_chunk=dc.kv_chunk if kv_chunk is None else kv_chunk, workspace=workspace, out=out)


def ref_decode(dc, window=None, k_cache=None, v_cache=None):
    return oracle.decode(bits(dc.q), bits(dc.k_cache if k_cache is None else k_cache),
                         bits(dc.v_cache if v_cache is None else v_cache), dc.page_table.numpy(),
                         dc.seq_lens.numpy(), None if dc.sinks is None else dc.sinks.numpy(),
                         window=dc.window if window is None else window, scale=dc.scale)


def assert_clean_device():
    st, b = sa.sink_attn_read_device_error()
    assert st == 0, f"device error word {b:#x}"


LENS = [1, 15, 16, 17, 255, 1023, 1024, 1025, 2049, 4000, 0, 333]

CASES = {
    "G8 D64 chunk1024": dict(lens=LENS, hq=64, hkv=8, d=64, chunk=1024),
    "G8 D64 chunk64 (many chunks)": dict(lens=LENS, hq=64, hkv=8, d=64, chunk=64),
    "G8 D64 chunk16": dict(lens=[1, 16, 17, 100, 513], hq=16, hkv=2, d=64, chunk=16),
    "G8 D64 W128": dict(lens=LENS, hq=64, hkv=8, d=64, chunk=1024, window=128),
    "G8 D64 W1": dict(lens=LENS, hq=16, hkv=2, d=64, chunk=1024, window=1),
    "G8 D64 W1500 chunk512": dict(lens=LENS, hq=16, hkv=2, d=64, chunk=512, window=1500),
    "G8 D64 sinks -inf": dict(lens=LENS, hq=16, hkv=2, d=64, chunk=1024, sinks="-inf"),
    "G8 D64 no sinks": dict(lens=LENS, hq=16, hkv=2, d=64, chunk=256, sinks=None),
    "G1 D64": dict(lens=LENS, hq=4, hkv=4, d=64, chunk=512),
    "G4 D128": dict(lens=LENS, hq=16, hkv=4, d=128, chunk=1024),
    "G16 D128 (Qwen3-235B-style)": dict(lens=LENS, hq=64, hkv=4, d=128, chunk=1024),
    "G16 D64 chunk128": dict(lens=LENS, hq=32, hkv=2, d=64, chunk=128),
    "G2 D128 W300": dict(lens=LENS, hq=4, hkv=2, d=128, chunk=128, window=300),
    "G16 D128 W100 chunk256": dict(lens=LENS, hq=32, hkv=2, d=128, chunk=256, window=100),
    # groups between 8 and 16: the second head tile is partly padding
    "G12 D128 chunk512": dict(lens=LENS, hq=24, hkv=2, d=128, chunk=512),
    "G10 D64 chunk256": dict(lens=LENS, hq=20, hkv=2, d=64, chunk=256),
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(name):
    c = CASES[name]
    dc = wl.decode_case(c["lens"], c["hq"], c["hkv"], c["d"], sinks=c.get("sinks", "normal"),
                        window=c.get("window", 0), seed=list(CASES).index(name), kv_chunk=c["chunk"],
                        spare_pages=5)
    got = gpu_decode(dc)
    assert_parity(got, ref_decode(dc), name)
    assert_clean_device()


def test_decode_nan_in_unused_slots():
    """Cache positions past each sequence's end (inside its last page) and before a
    window's start hold NaN: they must not reach the output."""
    dc = wl.decode_case([17, 1000, 1025, 31], 16, 2, 64, seed=21, kv_chunk=256)
    P = 16
    kc, vc = dc.k_cache.clone(), dc.v_cache.clone()
    for b in range(dc.batch):
        L = int(dc.seq_lens[b])
        last = int(dc.page_table[b, (L - 1) // P])
        used = L - ((L - 1) // P) * P
        kc[last, :, used:] = float("nan")
        vc[last, :, used:] = float("nan")
    got = gpu_decode(dc, k_cache=kc, v_cache=vc)
    assert_parity(got, ref_decode(dc, k_cache=kc, v_cache=vc), "NaN past the end")
    # window start inside a page: positions before it are NaN as well
    W = 100
    kc2, vc2 = kc.clone(), vc.clone()
    for b in range(dc.batch):
        L = int(dc.seq_lens[b])
        lo = max(0, L - W)
        for t in range(0, lo):
            pg = int(dc.page_table[b, t // P])
            kc2[pg, :, t % P] = float("nan")
            vc2[pg, :, t % P] = float("nan")
    got = gpu_decode(dc, window=W, k_cache=kc2, v_cache=vc2)
    ref = ref_decode(dc, window=W, k_cache=kc2, v_cache=vc2)
    assert_parity(got, ref, "NaN before the window")
    assert_clean_device()


def test_decode_guard_bands():
    """Guard rows around `out` and guard bytes after the workspace are untouched."""
    dc = wl.decode_case([3000, 5, 2048], 16, 2, 64, seed=22, kv_chunk=512)
    B = dc.batch
    g = 8
    big = torch.full((B + 2 * g, 16, 64), 3.5, dtype=torch.bfloat16, device="cuda")
    need = sa.sink_attn_decode_workspace_bytes(B, 16, 64, dc.max_seq_len, 512)
    assert need > 0
    ws_big = torch.full((need + 4096,), 0xA5, dtype=torch.uint8, device="cuda")
    got = gpu_decode(dc, out=big[g:g + B], workspace=ws_big[:need])
    assert torch.all(big[:g] == 3.5) and torch.all(big[g + B:] == 3.5)
    assert torch.all(ws_big[need:] == 0xA5)
    assert_parity(got, ref_decode(dc), "guarded")
    assert_clean_device()


def test_decode_workspace_reuse_without_clearing():
    """The workspace needs no initialisation: garbage in it does not change the result."""
    dc = wl.decode_case([2500, 700], 16, 2, 64, seed=23, kv_chunk=256)
    need = sa.sink_attn_decode_workspace_bytes(2, 16, 64, dc.max_seq_len, 256)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN patterns
    a = gpu_decode(dc, workspace=ws)
    b = gpu_decode(dc, workspace=ws)
    assert torch.equal(a, b)
    assert_parity(a, ref_decode(dc), "dirty workspace")


def test_decode_zero_length_and_empty_batch():
    dc = wl.decode_case([0, 0, 5], 8, 1, 64, seed=24)
    got = gpu_decode(dc)
    assert torch.count_nonzero(got[:2].float()) == 0
    assert_parity(got, ref_decode(dc), "zero lengths")
    dz = wl.decode_case([0, 0], 8, 1, 64, seed=25)
    got = gpu_decode(dz, max_seq_len=0)
    assert torch.count_nonzero(got.float()) == 0
    assert_clean_device()


def test_decode_bad_page_id_reported_not_faulted():
    dc = wl.decode_case([40, 40], 8, 1, 64, seed=26)
    pt = dc.page_table.clone()
    pt[1, 1] = dc.k_cache.shape[0] + 100  # outside the pool
    gpu_decode(dc, page_table=pt)
    st, b = sa.sink_attn_read_device_error()
    assert st == 5 and (b & 0x4)


def test_decode_seq_len_over_bound_reported():
    dc = wl.decode_case([40, 40], 8, 1, 64, seed=27)
    gpu_decode(dc, max_seq_len=32)
    st, b = sa.sink_attn_read_device_error()
    assert st == 5 and (b & 0x8)


def test_decode_host_validation():
    dc = wl.decode_case([40], 8, 1, 64, seed=28)
    with pytest.raises(sa.SinkAttnError) as e:
        gpu_decode(dc, kv_chunk=100)  # not a multiple of the page size
    assert e.value.status == 1
    with pytest.raises(sa.SinkAttnError) as e:
        sa.sink_attn_decode(dc.q.cuda(), dc.k_cache.cuda(), dc.v_cache.cuda(), dc.page_table.cuda(),
                            dc.seq_lens.cuda(), dc.sinks.cuda(), 5000, kv_chunk=1024,
                            workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 3


# ---------------------------------------------------------------------------
# Full-size workloads.
# ---------------------------------------------------------------------------

def test_decode_gptoss_full_size():
    """Batch 64, contexts U[1024, 8192], 64/8 heads, chunks of 1024: every output."""
    dc = wl.gptoss_decode(0)
    got = gpu_decode(dc)
    assert_parity(got, ref_decode(dc), dc.name, strict=True)
    assert_clean_device()


def test_decode_qwen_full_size():
    """Qwen3-235B-style decode (64/4 heads, group of 16, head_dim 128): every output."""
    dc = wl.qwen_decode(0)
    got = gpu_decode(dc)
    assert_parity(got, ref_decode(dc), dc.name, strict=True)
    assert_clean_device()


def test_decode_long_context_full_size_sampled():
    """Batch 128 x 32768 (8.6 GB of K/V), full and 128-window calls alternating on the
    same cache; the sampled sequences (drawn on the CPU) against the oracle."""
    sample = [0, 41, 127]
    dc = wl.long_decode(0, window=0, cache_device="cuda", only_seqs=sample)
    outs = []
    for w in (0, 128, 0, 128):
        outs.append(gpu_decode(dc, window=w).cpu())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[2]) and torch.equal(outs[1], outs[3])
    # the oracle gets a compact CPU cache holding only the sampled sequences' pages
    P = 16
    npg = 32768 // P
    kc = torch.empty((len(sample) * npg, 8, P, 64), dtype=torch.bfloat16)
    vc = torch.empty_like(kc)
    pt = torch.empty((len(sample), npg), dtype=torch.int32)
    for i, b in enumerate(sample):
        kb, vb = wl.draw_seq_kv(0, b, npg, 8, 64)
        kc[i * npg:(i + 1) * npg] = kb
        vc[i * npg:(i + 1) * npg] = vb
        pt[i] = torch.arange(i * npg, (i + 1) * npg, dtype=torch.int32)
    q = dc.q[sample]
    sl = torch.full((len(sample),), 32768, dtype=torch.int32)
    for w, got in ((0, outs[0]), (128, outs[1])):
        ref = oracle.decode(bits(q), bits(kc), bits(vc), pt.numpy(), sl.numpy(), dc.sinks.numpy(),
                            window=w, scale=dc.scale)
        assert_parity(got[sample], ref, f"long decode window {w}", strict=True)
    del dc
    torch.cuda.empty_cache()
    assert_clean_device()


def test_decode_graph_capture_matches_direct_call():
    """Split + merge captured in one CUDA graph (the PDL merge launch included) give the
    same bits as the direct call; replay after new page-table and length values too."""
    dc = wl.gptoss_decode(0)
    dq, dk, dv = dc.q.cuda(), dc.k_cache.cuda(), dc.v_cache.cuda()
    dpt, dsl, dsk = dc.page_table.cuda(), dc.seq_lens.cuda(), dc.sinks.cuda()
    need = sa.sink_attn_decode_workspace_bytes(dc.batch, dc.num_q_heads, dc.head_dim,
                                               dc.max_seq_len, dc.kv_chunk)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(dq)

    def call(stream):
        sa.sink_attn_decode(dq, dk, dv, dpt, dsl, dsk, dc.max_seq_len, scale=dc.scale,
                            kv_chunk=dc.kv_chunk, workspace=ws, out=out, stream=stream)

    call(None)
    direct = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(torch.cuda.current_stream())
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, direct)
    # new lengths written into the captured buffers between replays
    dsl.copy_(torch.clamp(dc.seq_lens - 999, min=1).cuda())
    g.replay()
    torch.cuda.synchronize()
    dc2 = wl.DecodeCase(dc.q, dc.k_cache, dc.v_cache, dc.page_table,
                        torch.clamp(dc.seq_lens - 999, min=1), dc.sinks, 0, dc.scale)
    assert_parity(out, ref_decode(dc2), "graph replay, shorter lengths", strict=True)
    assert_clean_device()


@pytest.mark.parametrize("hq,hkv,d", [(16, 2, 64), (64, 4, 128)])
def test_decode_wait_timeout_reported_then_clean(hq, hkv, d):
    """A pipeline wait that runs out: the test switch withholds the copy of one page (chunk 0,
    kv head 0, sequence 0), so its consumers' bounded wait gives up after 20 ms. The call
    returns, the device error word carries the timeout bit, every output outside the
    aborted CTA's heads is still right, and the next normal call in the same process is
    clean and matches the oracle."""
    dc = wl.decode_case([3000, 1500, 17, 2100], hq, hkv, d, seed=41, kv_chunk=1024)
    args = (dc.q.cuda(), dc.k_cache.cuda(), dc.v_cache.cuda(), dc.page_table.cuda(),
            dc.seq_lens.cuda(), dc.sinks.cuda(), dc.max_seq_len)
    ref = oracle.decode(bits(dc.q), bits(dc.k_cache), bits(dc.v_cache), dc.page_table.numpy(),
                        dc.seq_lens.numpy(), dc.sinks.numpy(), window=0, scale=dc.scale)
    sa.sink_attn_read_device_error()
    sa.sink_attn_debug_decode_withhold_page(True, 20_000_000)
    try:
        out = sa.sink_attn_decode(*args, window=0, scale=dc.scale, kv_chunk=1024)
        st, b = sa.sink_attn_read_device_error()
    finally:
        sa.sink_attn_debug_decode_withhold_page(False)
    assert st == 5 and (b & 0x1), f"status {st}, bits {b:#x}"
    G = hq // hkv
    keep = torch.ones(dc.batch, hq, dtype=torch.bool)
    keep[0, :G] = False  # the heads the aborted CTA serves
    got = out.float().cpu()
    assert_parity(got[keep], ref[keep.numpy()], "outside the aborted CTA", strict=True)
    out = sa.sink_attn_decode(*args, window=0, scale=dc.scale, kv_chunk=1024)
    assert_clean_device()
    assert_parity(out, ref, "next call", strict=True)
