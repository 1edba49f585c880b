"""GPU tests of the paged cache path: sink_attn_append_kv (bit-exact placement of the new
rows) and sink_attn_prefill_paged (chunked prefill: new query rows against everything
cached before them plus themselves) against the fp64 oracle. Every cache slot that holds
no token is a bf16 NaN, so any masked position whose value reaches a sum shows up."""
import numpy as np
import pytest
import torch

import gqa_attention_head_gb300 as sa
import oracle
from gqa_attention_head_gb300 import workloads as wl
from parity import assert_parity

pytestmark = pytest.mark.gpu

bits = wl.bf16_bits
LSE_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    from gqa_attention_head_gb300 import _build
    _build.build()
    sa.load_library()
    sa.sink_attn_read_device_error()
    yield


def assert_clean_device():
    st, b = sa.sink_attn_read_device_error()
    assert st == 0, f"device error word {b:#x}"


def expected_cache_after_append(pc):
    kc, vc = pc.k_cache.clone(), pc.v_cache.clone()
    cu = pc.cu_seqlens.tolist()
    for s, L0 in enumerate(pc.prefix_lens):
        for i in range(pc.new_lens[s]):
            pos = L0 + i
            pid = int(pc.page_table[s, pos // 16])
            kc[pid, :, pos % 16] = pc.k_new[cu[s] + i]
            vc[pid, :, pos % 16] = pc.v_new[cu[s] + i]
    return kc, vc


def test_append_kv_bit_exact():
    gen = torch.Generator().manual_seed(500)
    for d in (64, 128):
        pc = wl.paged_prefill_case([0, 3, 16, 100, 31], [7, 13, 16, 1, 300], 8, 4, d, gen=gen)
        kc, vc = pc.k_cache.cuda(), pc.v_cache.cuda()
        sa.sink_attn_append_kv(pc.k_new.cuda(), pc.v_new.cuda(), kc, vc, pc.page_table.cuda(),
                               pc.cu_seqlens.cuda(), pc.seq_lens.cuda())
        ek, ev = expected_cache_after_append(pc)
        # compare bit patterns (NaN slots included)
        assert torch.equal(kc.cpu().view(torch.int16), ek.view(torch.int16))
        assert torch.equal(vc.cpu().view(torch.int16), ev.view(torch.int16))
        assert_clean_device()


CASES = {
    "D64 G8 prefixes": dict(pre=[0, 1, 15, 16, 17, 127, 128, 129, 1000],
                            new=[5, 128, 129, 1, 300, 64, 17, 200, 130], hq=16, hkv=2, d=64),
    "D64 G8 W100": dict(pre=[0, 90, 300, 7], new=[250, 40, 129, 1], hq=16, hkv=2, d=64, window=100),
    "D64 no sinks G1": dict(pre=[33, 0], new=[70, 9], hq=4, hkv=4, d=64, sinks=None),
    "D64 sinks -inf G3": dict(pre=[50], new=[200], hq=6, hkv=2, d=64, sinks="-inf"),
    "D128 G16": dict(pre=[0, 129, 500], new=[140, 64, 257], hq=32, hkv=2, d=128),
    "D128 G4 W64": dict(pre=[200, 10], new=[100, 300], hq=8, hkv=2, d=128, window=64),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_paged(name):
    c = CASES[name]
    gen = torch.Generator().manual_seed(600 + list(CASES).index(name))
    pc = wl.paged_prefill_case(c["pre"], c["new"], c["hq"], c["hkv"], c["d"],
                               sinks=c.get("sinks", "normal"), window=c.get("window", 0), gen=gen)
    ref_o, ref_l = oracle.prefill_paged(bits(pc.q), bits(pc.k_new), bits(pc.v_new),
                                        bits(pc.k_cache), bits(pc.v_cache), pc.page_table.numpy(),
                                        pc.cu_seqlens.numpy(), pc.seq_lens.numpy(),
                                        None if pc.sinks is None else pc.sinks.numpy(),
                                        window=pc.window, scale=pc.scale, with_lse=True)
    kc, vc = pc.k_cache.cuda(), pc.v_cache.cuda()
    out, lse = sa.sink_attn_prefill_paged(
        pc.q.cuda(), pc.k_new.cuda(), pc.v_new.cuda(), kc, vc, pc.page_table.cuda(),
        pc.cu_seqlens.cuda(), pc.seq_lens.cuda(), None if pc.sinks is None else pc.sinks.cuda(),
        pc.max_q_len, pc.max_seq_len, window=pc.window, scale=pc.scale, want_lse=True)
    assert_parity(out, ref_o, name)
    got_l = lse.cpu().double().numpy()
    assert np.all(np.isfinite(got_l)) and np.abs(got_l - ref_l).max() <= LSE_ABS, name
    ek, ev = expected_cache_after_append(pc)
    assert torch.equal(kc.cpu().view(torch.int16), ek.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), ev.view(torch.int16))
    assert_clean_device()


@pytest.mark.parametrize("d,window", [(64, 0), (64, 200), (128, 0)])
def test_chunked_prefill_end_to_end(d, window):
    """Each sequence is prefilled in three chunks through sink_attn_prefill_paged, the
    cache growing on the GPU; all outputs against the oracle's one-pass prefill."""
    gen = torch.Generator().manual_seed(700 + d + window)
    lengths = [700, 129, 1000]
    hq, hkv = 16, 2
    case = wl.prefill_case(lengths, hq, hkv, d, sinks="normal", window=window, gen=gen)
    ref = oracle.prefill(bits(case.q), bits(case.k), bits(case.v), case.sinks.numpy(),
                         case.cu_seqlens.numpy(), window=window, scale=case.scale)
    P = 16
    npg = [(L + P - 1) // P for L in lengths]
    total = sum(npg) + 4
    perm = torch.randperm(total, generator=gen).to(torch.int32)
    pt = torch.full((len(lengths), max(npg)), -1, dtype=torch.int32)
    at = 0
    for s, n in enumerate(npg):
        pt[s, :n] = perm[at:at + n]
        at += n
    nan = torch.tensor([wl.BF16_NAN], dtype=torch.int16).view(torch.bfloat16)
    kc = nan.repeat(total * hkv * P * d).view(total, hkv, P, d).cuda()
    vc = kc.clone()
    ptd, sk = pt.cuda(), case.sinks.cuda()
    cu = case.cu_seqlens.tolist()
    splits = [[0, 100, 400, 700], [0, 1, 2, 129], [0, 513, 640, 1000]]
    got = torch.empty_like(case.q)
    for c in range(3):
        rows, new_lens, seq_lens = [], [], []
        for s in range(len(lengths)):
            a, b = splits[s][c], splits[s][c + 1]
            rows.extend(range(cu[s] + a, cu[s] + b))
            new_lens.append(b - a)
            seq_lens.append(b)
        rows_t = torch.tensor(rows, dtype=torch.int64)
        ncu = torch.tensor(np.concatenate([[0], np.cumsum(new_lens)]), dtype=torch.int32)
        out, _ = sa.sink_attn_prefill_paged(
            case.q[rows_t].cuda(), case.k[rows_t].cuda(), case.v[rows_t].cuda(), kc, vc, ptd,
            ncu.cuda(), torch.tensor(seq_lens, dtype=torch.int32).cuda(), sk, max(new_lens),
            max(seq_lens), window=window, scale=case.scale)
        got[rows_t] = out.cpu()
    assert_parity(got, ref, f"chunked prefill D{d} W{window}", strict=True)
    assert_clean_device()


def test_prefill_paged_bad_page_id_recorded():
    gen = torch.Generator().manual_seed(800)
    pc = wl.paged_prefill_case([40, 10], [30, 20], 8, 1, 64, gen=gen)
    pt = pc.page_table.clone()
    pt[0, 1] = pc.k_cache.shape[0] + 5  # out of range (covers cached positions 16..31)
    kc, vc = pc.k_cache.cuda(), pc.v_cache.cuda()
    out, _ = sa.sink_attn_prefill_paged(
        pc.q.cuda(), pc.k_new.cuda(), pc.v_new.cuda(), kc, vc, pt.cuda(), pc.cu_seqlens.cuda(),
        pc.seq_lens.cuda(), pc.sinks.cuda(), pc.max_q_len, pc.max_seq_len, scale=pc.scale)
    st, b = sa.sink_attn_read_device_error()
    assert st == 5 and (b & 0x4), f"expected the page-id bit, got {b:#x}"
    # the other sequence is unaffected
    ref = oracle.prefill_paged(bits(pc.q), bits(pc.k_new), bits(pc.v_new), bits(pc.k_cache),
                               bits(pc.v_cache), pc.page_table.numpy(), pc.cu_seqlens.numpy(),
                               pc.seq_lens.numpy(), pc.sinks.numpy(), scale=pc.scale)
    assert_parity(out[30:], ref[30:], "sequence with valid pages")


def test_chunked_prefill_full_size_every_element():
    """The gpt-oss chunked-prefill workload (4 sequences, 2048 new rows each on top of
    U[2048, 6144] cached tokens) in the launch configuration that is timed, against the
    oracle's paged prefill on every (row, head, d) of the output at the strict bound, and
    every row's log-sum-exp within 1e-3."""
    pc = wl.gptoss_chunked_prefill(seed=0)
    kc, vc = pc.k_cache.cuda(), pc.v_cache.cuda()
    out, lse = sa.sink_attn_prefill_paged(
        pc.q.cuda(), pc.k_new.cuda(), pc.v_new.cuda(), kc, vc, pc.page_table.cuda(),
        pc.cu_seqlens.cuda(), pc.seq_lens.cuda(), pc.sinks.cuda(), pc.max_q_len, pc.max_seq_len,
        scale=pc.scale, want_lse=True)
    torch.cuda.synchronize()
    assert_clean_device()
    ref, ref_lse = oracle.prefill_paged(bits(pc.q), bits(pc.k_new), bits(pc.v_new),
                                        bits(pc.k_cache), bits(pc.v_cache),
                                        pc.page_table.numpy(), pc.cu_seqlens.numpy(),
                                        pc.seq_lens.numpy(), pc.sinks.numpy(), window=0,
                                        scale=pc.scale, with_lse=True)
    assert_parity(out, ref, "chunked prefill, every output", strict=True)
    got_lse = lse.cpu().numpy()
    assert np.all(np.isfinite(got_lse))
    assert np.max(np.abs(got_lse - ref_lse)) <= 1e-3
