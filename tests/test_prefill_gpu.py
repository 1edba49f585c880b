"""GPU parity of sink_attn_prefill (tcgen05 kernel, called through the C ABI) against the
fp64 oracle, element by element, on seeded inputs; plus edge cases, guard bands and
the device-side checks."""
import ctypes

import numpy as np
import pytest
import torch

import gqa_attention_head_gb300 as sa
import oracle
from gqa_attention_head_gb300 import workloads as wl
from parity import assert_parity, to_f64

pytestmark = pytest.mark.gpu

bits = wl.bf16_bits


@pytest.fixture(scope="module", autouse=True)
def _library():
    from gqa_attention_head_gb300 import _build
    _build.build()
    sa.load_library()
    sa.sink_attn_read_device_error()  # start from a clear error word
    yield


def gpu_prefill(case, out=None, window=None, max_seqlen=None, cu=None):
    return sa.sink_attn_prefill(
        case.q.cuda(), case.k.cuda(), case.v.cuda(),
        None if case.sinks is None else case.sinks.cuda(),
        (case.cu_seqlens if cu is None else cu).cuda(),
        case.max_seqlen if max_seqlen is None else max_seqlen,
        window=case.window if window is None else window, scale=case.scale, out=out)


def ref_prefill(case, window=None):
    return oracle.prefill(bits(case.q), bits(case.k), bits(case.v),
                          None if case.sinks is None else case.sinks.numpy(),
                          case.cu_seqlens.numpy(), window=case.window if window is None else window,
                          scale=case.scale)


def assert_clean_device():
    st, b = sa.sink_attn_read_device_error()
    assert st == 0, f"device error word {b:#x}"


def valid_rows(case):
    cu = case.cu_seqlens.tolist()
    return np.concatenate([np.arange(cu[s], cu[s + 1]) for s in range(len(cu) - 1)] or
                          [np.zeros(0, np.int64)]).astype(np.int64)


CASES = {
    "tiny 1x256 Hq8/Hkv1 D64": lambda: wl.tiny_prefill(0),
    "ragged D64 G4 causal": lambda: wl.prefill_case([1, 127, 128, 129, 300, 0, 513], 8, 2, 64, seed=1),
    "ragged D64 G4 W128": lambda: wl.prefill_case([1, 127, 128, 129, 300, 0, 513], 8, 2, 64,
                                                  window=128, seed=1),
    "ragged D64 W1": lambda: wl.prefill_case([5, 130, 257], 4, 2, 64, window=1, seed=2),
    "ragged D64 W200": lambda: wl.prefill_case([150, 700], 4, 1, 64, window=200, seed=3),
    "D64 MHA G1 no sinks": lambda: wl.prefill_case([255, 256, 33], 4, 4, 64, sinks=None, seed=4),
    "D64 sinks -inf": lambda: wl.prefill_case([400], 8, 1, 64, sinks="-inf", seed=5),
    "D128 G8 sinks -inf": lambda: wl.prefill_case([200, 385], 8, 1, 128, sinks="-inf", seed=6),
    "D128 G8 sinks N(0,1)": lambda: wl.prefill_case([200, 385], 8, 1, 128, seed=6),
    "D128 G16 W64": lambda: wl.prefill_case([260, 64, 1], 16, 1, 128, window=64, seed=7),
    "D128 G4 W1000 ragged": lambda: wl.prefill_case([1000, 1001, 77], 8, 2, 128, window=1000, seed=8),
    # the bound on units per CTA (every q tile of the longest sequence in every sequence,
    # 32 x 100 x 8 x 4 / 152 = 674) exceeds the 512 the shared-memory unit list holds:
    # head_dim 64 then decodes each unit when it starts
    "100 sequences, one of 4096, D64 G8": lambda: wl.prefill_case(
        [4096] + [int(x) for x in np.random.default_rng(17).integers(1, 100, 99)], 64, 8, 64,
        seed=17),
    "100 sequences, one of 4096, D128 G8": lambda: wl.prefill_case(
        [4096] + [int(x) for x in np.random.default_rng(18).integers(1, 100, 99)], 64, 8, 128,
        seed=18),
    # more sequences than the snake schedule's tables hold: round-robin over all unit ids
    "130 sequences D64 G2": lambda: wl.prefill_case(
        [int(x) for x in np.random.default_rng(16).integers(0, 200, 130)], 4, 2, 64, seed=16),
    # short windows at head_dim 64 with groups of 8k query heads: the kernel whose unit is 32
    # queries x 8 heads over one 160-key span (lengths around its 32-row blocks, spans that
    # reach into the previous sequence or before the first row, empty sequences)
    "band D64 G8 W128 ragged": lambda: wl.prefill_case(
        [1, 31, 32, 33, 127, 128, 129, 300, 0, 513], 16, 2, 64, window=128, seed=21),
    "band D64 G8 W1": lambda: wl.prefill_case([5, 130, 257], 8, 1, 64, window=1, seed=22),
    "band D64 G16 W100": lambda: wl.prefill_case([260, 64, 1, 97], 32, 2, 64, window=100,
                                                 seed=23),
    "band D64 G8 W33 no sinks": lambda: wl.prefill_case([200, 45], 8, 1, 64, window=33,
                                                        sinks=None, seed=24),
    "band D64 G8 W128 sinks -inf": lambda: wl.prefill_case([400], 8, 1, 64, window=128,
                                                           sinks="-inf", seed=25),
    "band 300 sequences D64 G8 W64": lambda: wl.prefill_case(
        [int(x) for x in np.random.default_rng(26).integers(0, 200, 300)], 8, 1, 64, window=64,
        seed=26),
    # the last window the short-window kernel takes, and the first it leaves to the general one
    "band D64 G8 W127": lambda: wl.prefill_case([300, 129, 1], 8, 1, 64, window=127, seed=27),
    "D64 G8 W129 (general kernel)": lambda: wl.prefill_case([300, 129, 1], 8, 1, 64, window=129,
                                                            seed=28),
    # as many sequences as the short-window kernel's sequence table holds
    "band 1024 sequences D64 G8 W128": lambda: wl.prefill_case(
        [int(x) for x in np.random.default_rng(29).integers(0, 40, 1024)], 8, 1, 64, window=128,
        seed=29),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_matches_oracle(name):
    case = CASES[name]()
    got = gpu_prefill(case)
    ref = ref_prefill(case)
    rows = valid_rows(case)
    assert_parity(got[rows], ref[rows], name, strict=name.startswith("tiny"))
    assert_clean_device()


def test_prefill_rescale_path():
    """Key norms grow along the sequence so the running maximum keeps jumping by more
    than 2^8: exercises the O rescale between PV steps."""
    case = wl.prefill_case([700, 333], 8, 2, 64, seed=9)
    T = case.total_tokens
    growth = (1.0 + torch.arange(T, dtype=torch.float32) / 40.0).view(T, 1, 1)
    case.k = (case.k.float() * growth).to(torch.bfloat16)
    case.q = (case.q.float() * 3.0).to(torch.bfloat16)
    got = gpu_prefill(case)
    assert_parity(got, ref_prefill(case), "rescale path")
    assert_clean_device()


@pytest.mark.parametrize("hkv,window", [(2, 0), (1, 128)])
def test_prefill_large_sink_gives_zero(hkv, window):
    case = wl.prefill_case([300, 50], 8, hkv, 64, sinks=1.0e4, window=window, seed=10)
    got = gpu_prefill(case)
    assert torch.count_nonzero(got.float()) == 0
    assert_clean_device()


@pytest.mark.parametrize("hkv,window", [(2, 0), (1, 128)])
def test_prefill_guard_bands_and_foreign_rows_untouched(hkv, window):
    """Rows of tokens outside every sequence, and guard rows around `out`, keep their
    sentinel: the kernel writes only the rows it owns."""
    case = wl.prefill_case([129, 40], 8, hkv, 64, window=window, seed=11, extra_tokens=7)
    T = case.total_tokens
    guard = 64
    big = torch.full((T + 2 * guard, 8, 64), -7.25, dtype=torch.bfloat16, device="cuda")
    out = big[guard:guard + T]
    gpu_prefill(case, out=out)
    assert torch.all(big[:guard] == -7.25) and torch.all(big[guard + T:] == -7.25)
    assert torch.all(out[169:] == -7.25)
    rows = valid_rows(case)
    assert_parity(out[rows], ref_prefill(case)[rows], "guarded")
    assert_clean_device()


@pytest.mark.parametrize("d,window,hkv", [(64, 0, 2), (128, 0, 2), (64, 128, 2), (128, 50, 2),
                                           (64, 128, 1)])
def test_prefill_out_16_byte_aligned_matches_32_byte_aligned(d, window, hkv):
    """Output rows go out as 32-byte stores when `out` is 32-byte aligned, as 16-byte stores
    when it is only 16-byte aligned (what the interface requires): the two give the same
    bits, and the bytes around the offset buffer keep their sentinel. Windowed head_dim 64
    runs the kernel form whose epilogue is deferred into the next unit (groups of 4) or the
    short-window kernel (groups of 8)."""
    case = wl.prefill_case([129, 300, 40], 8, hkv, d, window=window, seed=13, extra_tokens=5)
    n = case.total_tokens * 8 * d
    ref = gpu_prefill(case)
    assert ref.data_ptr() % 32 == 0
    flat = torch.full((n + 32,), -7.25, dtype=torch.bfloat16, device="cuda")
    out = flat[8:8 + n].view(case.total_tokens, 8, d)  # 16 bytes past a 256-byte boundary
    assert out.data_ptr() % 32 == 16
    gpu_prefill(case, out=out)
    rows = valid_rows(case)
    assert np.array_equal(bits(out[rows]), bits(ref[rows]))
    assert torch.all(flat[:8] == -7.25) and torch.all(flat[8 + n:] == -7.25)
    assert_parity(out[rows], ref_prefill(case)[rows], f"16-byte aligned out D{d} W{window}")
    assert_clean_device()


def test_prefill_empty_inputs_are_noops():
    case = wl.prefill_case([0, 0], 4, 2, 64, seed=12, extra_tokens=3)
    out = torch.full_like(case.q.cuda(), 1.5)
    gpu_prefill(case, out=out)
    assert torch.all(out == 1.5)
    assert_clean_device()


@pytest.mark.parametrize("hq,hkv,window", [(4, 2, 0), (8, 1, 128)])
def test_prefill_bad_cu_seqlens_reported_not_faulted(hq, hkv, window):
    """(8, 1, 128) runs the short-window kernel."""
    case = wl.prefill_case([64, 64], hq, hkv, 64, window=window, seed=13)
    bad = torch.tensor([0, 64, 1000], dtype=torch.int32)  # past total_tokens
    out = torch.zeros_like(case.q.cuda())
    gpu_prefill(case, out=out, cu=bad)
    st, b = sa.sink_attn_read_device_error()
    assert st == 5 and (b & 0x2)
    # the valid first sequence is still computed
    ref = ref_prefill(case)
    assert_parity(out[:64], ref[:64], "first sequence")


@pytest.mark.parametrize("hq,hkv,window", [(4, 2, 0), (8, 1, 128)])
def test_prefill_max_seqlen_too_small_reported(hq, hkv, window):
    case = wl.prefill_case([300], hq, hkv, 64, window=window, seed=14)
    gpu_prefill(case, max_seqlen=128)
    st, b = sa.sink_attn_read_device_error()
    assert st == 5 and (b & 0x2)


def test_prefill_host_validation():
    case = wl.prefill_case([16], 4, 3, 64, seed=15)
    with pytest.raises(sa.SinkAttnError) as e:
        gpu_prefill(case)  # 4 query heads, 3 kv heads
    assert e.value.status == 1
    case = wl.prefill_case([16], 4, 2, 96, seed=15)
    with pytest.raises(sa.SinkAttnError) as e:
        gpu_prefill(case)
    assert e.value.status == 2


# ---------------------------------------------------------------------------
# Full-size workloads. The four named prefill workloads are compared with the oracle on
# every output element (the oracle takes tens of seconds per workload on the host cores);
# the two 32768-token sequences, too long for that, on sampled rows (first/last rows of
# every sequence, tile boundaries, and random rows) plus a property that holds everywhere.
# ---------------------------------------------------------------------------

def sample_rows(case, n_random, seed):
    g = np.random.default_rng(seed)
    cu = case.cu_seqlens.tolist()
    toks = []
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        L = b - a
        for i in [0, 1, 127, 128, 129, L // 2, L - 129, L - 128, L - 2, L - 1]:
            if 0 <= i < L:
                toks.append(a + i)
    toks += list(g.integers(0, case.total_tokens, n_random))
    toks = np.array(sorted(set(toks)), dtype=np.int64)
    heads = g.integers(0, case.num_q_heads, len(toks)).astype(np.int32)
    # every head at the last token of the longest sequence
    s_long = int(np.argmax(case.lengths))
    last = cu[s_long + 1] - 1
    toks = np.concatenate([toks, np.full(case.num_q_heads, last)])
    heads = np.concatenate([heads, np.arange(case.num_q_heads, dtype=np.int32)])
    return toks, heads


FULL = {
    "gpt-oss prefill causal": lambda: wl.gptoss_prefill(0, window=0),
    "gpt-oss prefill W128": lambda: wl.gptoss_prefill(0, window=128),
    "Qwen3-235B prefill sinks -inf": lambda: wl.qwen_prefill(0, sinks="-inf"),
    "Qwen3-235B prefill sinks N(0,1)": lambda: wl.qwen_prefill(0, sinks="normal"),
}


@pytest.mark.parametrize("name", list(FULL))
def test_prefill_full_size_every_element(name):
    """Every (token, head, d) of a named full-size workload against the fp64 oracle, at the
    strict bound over the whole tensor: the late units of the snake schedule, the deferred
    epilogues across unit boundaries and the rescales of long rows are all covered."""
    case = FULL[name]()
    got = gpu_prefill(case)
    torch.cuda.synchronize()
    assert_clean_device()
    ref = ref_prefill(case)
    assert_parity(got, ref, name, strict=True)


LONG = {
    # the longest single sequences: 256 q tiles x 256 key tiles in one causal unit chain
    "one 32768-token sequence D64 G8 causal": lambda: wl.prefill_case([32768], 64, 8, 64,
                                                                      seed=77),
    "one 32768-token sequence D128 G16 W128": lambda: wl.prefill_case([32768], 64, 4, 128,
                                                                      window=128, seed=78),
    # the short-window kernel over 1024 query blocks of one sequence
    "one 32768-token sequence D64 G8 W128": lambda: wl.prefill_case([32768], 64, 8, 64,
                                                                    window=128, seed=79),
}


@pytest.mark.parametrize("name", list(LONG))
def test_prefill_long_sequence_sampled(name):
    case = LONG[name]()
    got = gpu_prefill(case)
    torch.cuda.synchronize()
    assert torch.isfinite(got.float()).all()
    toks, heads = sample_rows(case, 1500, seed=1)
    ref = oracle.prefill_rows(bits(case.q), bits(case.k), bits(case.v),
                              None if case.sinks is None else case.sinks.numpy(),
                              case.cu_seqlens.numpy(), toks, heads, window=case.window,
                              scale=case.scale)
    got_rows = to_f64(got[torch.from_numpy(toks).cuda(), torch.from_numpy(heads).long().cuda()])
    assert_parity(got_rows, ref, name, strict=True)
    # property at full size: every output row lies in the convex hull bound of |v|
    vmax = case.v.float().abs().max().item()
    assert got.float().abs().max().item() <= vmax * (1 + 1e-2)
    assert_clean_device()


@pytest.mark.parametrize("d,window", [(64, 0), (128, 0), (64, 128)])
def test_nan_input_row_stays_local(d, window):
    """A NaN in one query row makes that row's output NaN and nothing else. The row's
    softmax state (max and sum) is NaN in only some lanes of a warp, so any warp-aligned
    step that takes a per-lane value as its condition would diverge here. Window 128 with
    groups of 8 runs the short-window kernel."""
    case = wl.prefill_case([300, 129], 16, 2, d, window=window, seed=900 + d)
    q = case.q.clone()
    q[7, 3, 5] = float("nan")
    got = sa.sink_attn_prefill(q.cuda(), case.k.cuda(), case.v.cuda(), case.sinks.cuda(),
                               case.cu_seqlens.cuda(), case.max_seqlen, window=window,
                               scale=case.scale)
    got = got.float().cpu()
    assert torch.isnan(got[7, 3]).all()
    rest = torch.ones(got.shape[:2], dtype=torch.bool)
    rest[7, 3] = False
    assert torch.isfinite(got[rest]).all()
    ref = ref_prefill(case)
    got[7, 3] = torch.from_numpy(ref[7, 3]).float()  # the NaN row was checked above
    assert_parity(got, ref, f"NaN query row D{d} W{window}")
    assert_clean_device()


@pytest.mark.parametrize("which", ["gpt-oss", "ragged with empty sequences"])
def test_prefill_from_host_matches_oracle(which):
    """The pipelined host-input prefill (row ranges cut across sequences, each a varlen call:
    copies in, kernel, copy out on three streams) against the oracle. Cutting a sequence
    moves its 128-row q-tile boundaries, which can change a per-warp rescale decision, so
    the bits may differ from one device-resident call but not beyond rounding."""
    if which == "gpt-oss":
        case = wl.gptoss_prefill(0, window=0)
        toks, heads = sample_rows(case, 1500, seed=3)
    else:
        case = wl.prefill_case([0, 300, 1, 0, 2000, 129, 40, 700], 16, 2, 64, window=200, seed=81)
        toks = valid_rows(case)
        toks = np.repeat(toks, case.num_q_heads)
        heads = np.tile(np.arange(case.num_q_heads, dtype=np.int32), len(toks) // case.num_q_heads)
    ref = oracle.prefill_rows(bits(case.q), bits(case.k), bits(case.v), case.sinks.numpy(),
                              case.cu_seqlens.numpy(), toks, heads, window=case.window,
                              scale=case.scale)
    hq, hk, hv = case.q.pin_memory(), case.k.pin_memory(), case.v.pin_memory()
    for kw in (dict(), dict(n_ranges=3, q_dev=torch.empty_like(case.q, device="cuda"),
                            k_dev=torch.empty_like(case.k, device="cuda"),
                            v_dev=torch.empty_like(case.v, device="cuda"),
                            out_dev=torch.empty_like(case.q, device="cuda"))):
        out = sa.sink_attn_prefill_from_host(hq, hk, hv, case.sinks, case.cu_seqlens,
                                             case.max_seqlen, window=case.window,
                                             scale=case.scale, **kw)
        torch.cuda.synchronize()
        got = out[torch.from_numpy(toks), torch.from_numpy(heads).long()]
        assert_parity(got, ref, f"from host {which} {sorted(kw)}", strict=True)
    assert_clean_device()

@pytest.mark.parametrize("d", [64, 128])
def test_prefill_from_host_one_range_equals_device_call(d):
    """One row range through the C pipeline, both copy directions on the compute stream
    (NULL copy streams): the varlen call then sees every sequence whole, so the output has
    the bits of sink_attn_prefill on device-resident inputs. Rows outside every sequence
    keep their sentinel in the host output."""
    case = wl.prefill_case([300, 0, 129, 1000, 1], 8, 2, d, seed=83, extra_tokens=6)
    ref = gpu_prefill(case).cpu()
    lib = sa.load_library()
    T, hq, _ = case.q.shape
    hq_, hk_, hv_ = case.q.pin_memory(), case.k.pin_memory(), case.v.pin_memory()
    hout = torch.full(case.q.shape, -7.25, dtype=torch.bfloat16).pin_memory()
    devs = [torch.empty_like(t, device="cuda") for t in (case.q, case.k, case.v, case.q)]
    cu = case.cu_seqlens.to(torch.int32).contiguous()
    sk = case.sinks.contiguous()
    S = cu.numel() - 1
    nb = int(lib.sink_attn_prefill_from_host_scratch_bytes(S, hq, 1))
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.sink_attn_prefill_from_host(
        p(hq_), p(hk_), p(hv_), p(sk), p(cu), S, T, hq, case.num_kv_heads, d, 0, case.scale,
        p(hout), *(p(t) for t in devs), p(scratch), nb, 1,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), None, None)
    assert st == 0
    torch.cuda.synchronize()
    rows = valid_rows(case)
    assert np.array_equal(bits(hout[rows]), bits(ref[rows]))
    assert torch.all(hout[case.cu_seqlens[-1].item():] == -7.25)
    assert_clean_device()


VARLEN = {
    "D64 G8": dict(m=[1, 500, 129, 7, 1000, 256], n=[1, 100, 129, 0, 300, 1], hq=16, hkv=2, d=64),
    "D64 G8 W100": dict(m=[300, 90, 1000], n=[250, 90, 3], hq=16, hkv=2, d=64, window=100),
    "D64 no sinks G1": dict(m=[200, 77], n=[64, 77], hq=4, hkv=4, d=64, sinks=None),
    "D128 G16": dict(m=[129, 700, 2000], n=[128, 257, 1000], hq=32, hkv=2, d=128),
    "D128 G4 W64": dict(m=[400, 50], n=[300, 50], hq=8, hkv=2, d=128, window=64),
}


def varlen_from_full(case, n):
    """Queries = the last n[s] rows of every full sequence; keys = all its rows."""
    cu = case.cu_seqlens.tolist()
    rows = np.concatenate([np.arange(cu[s + 1] - n[s], cu[s + 1]) for s in range(len(n))]
                          or [np.zeros(0, np.int64)]).astype(np.int64)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(n)]), dtype=torch.int32)
    return rows, cu_q


@pytest.mark.parametrize("name", list(VARLEN))
def test_prefill_varlen_matches_oracle(name):
    c = VARLEN[name]
    case = wl.prefill_case(c["m"], c["hq"], c["hkv"], c["d"], sinks=c.get("sinks", "normal"),
                           window=c.get("window", 0), seed=700 + list(VARLEN).index(name))
    rows, cu_q = varlen_from_full(case, c["n"])
    q = case.q[torch.from_numpy(rows)].contiguous()
    out, lse = sa.sink_attn_prefill_varlen(
        q.cuda(), case.k.cuda(), case.v.cuda(), None if case.sinks is None else case.sinks.cuda(),
        cu_q.cuda(), case.cu_seqlens.cuda(), max(c["n"]), max(c["m"]), window=case.window,
        scale=case.scale, want_lse=True)
    ref, ref_lse = oracle.prefill(bits(case.q), bits(case.k), bits(case.v),
                                  None if case.sinks is None else case.sinks.numpy(),
                                  case.cu_seqlens.numpy(), window=case.window, scale=case.scale,
                                  with_lse=True)
    assert_parity(out, ref[rows], name)
    got_lse = lse.cpu().numpy()
    fin = np.isfinite(ref_lse[rows])
    assert np.array_equal(np.isfinite(got_lse), fin)
    assert np.max(np.abs(got_lse[fin] - ref_lse[rows][fin]), initial=0.0) <= 1e-3
    assert_clean_device()


def test_prefill_varlen_equal_ranges_is_prefill_and_bad_lengths_reported():
    case = wl.prefill_case([300, 129, 1000], 16, 2, 64, seed=720)
    a = gpu_prefill(case)
    b, _ = sa.sink_attn_prefill_varlen(case.q.cuda(), case.k.cuda(), case.v.cuda(),
                                       case.sinks.cuda(), case.cu_seqlens.cuda(),
                                       case.cu_seqlens.cuda(), case.max_seqlen, case.max_seqlen,
                                       scale=case.scale)
    rows = torch.from_numpy(valid_rows(case))
    assert torch.equal(a.cpu()[rows].view(torch.int16), b.cpu()[rows].view(torch.int16))
    assert_clean_device()
    # a sequence with fewer keys than queries is skipped and reported, never read
    cu_k = torch.tensor([0, 300, 400, 1429], dtype=torch.int32)  # sequence 1: 100 keys, 129 q
    sa.sink_attn_prefill_varlen(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.sinks.cuda(),
                                case.cu_seqlens.cuda(), cu_k.cuda(), case.max_seqlen, 1029,
                                scale=case.scale)
    st, bits_ = sa.sink_attn_read_device_error()
    assert st == 5 and (bits_ & 0x8)
