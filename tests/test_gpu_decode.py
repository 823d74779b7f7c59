"""GPU parity: the CUDA path through the C ABI against the float64 oracle."""
import numpy as np
import pytest
import torch

from gpu_harness import GpuCase, compare, oracle_decode, torch_bf16_to_bits
from mla_paged_decode_02_gb300 import api, synth
from oracle import fp8_e4m3
from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu

BF, F8 = synth.KV_BF16, synth.KV_FP8_E4M3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    api.lib()


# ---------------------------------------------------------------- cache write
@pytest.mark.parametrize("kv", [BF, F8])
def test_cache_write_is_bit_exact(kv):
    case = synth.make_case(B=3, s_q=1, H=1, page_size=64, seq_lens=[1, 64, 300], seed=21, kv_dtype=kv)
    case.slot_mapping[5] = -1                       # a padding token is skipped
    g = GpuCase(case)
    ref = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits, case.slot_mapping,
                        case.page_size, kv, case.kv_scale)
    assert np.array_equal(g.cache_numpy(), ref)


@pytest.mark.parametrize("scale", [1.0, 3.0 / 448.0, 0.0071, 1.0e-3, 17.25, 2.0 ** -20])
def test_fp8_cache_write_exhaustive_over_bf16_inputs(scale):
    """Every one of the 65536 bf16 bit patterns goes through the quantising write."""
    all_bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    latent = all_bits.reshape(128, 512)
    rope = np.zeros((128, 64), dtype=np.uint16)
    slots = np.arange(128, dtype=np.int64)
    scale = float(np.float32(scale))
    lat_t = torch.from_numpy(latent.view(np.int16)).view(torch.bfloat16).cuda()
    rope_t = torch.from_numpy(rope.view(np.int16)).view(torch.bfloat16).cuda()
    cache = torch.full((2, 64, 576), 0x7F, dtype=torch.uint8, device="cuda")
    ks = torch.tensor([scale], dtype=torch.float32, device="cuda")
    api.cache_write(lat_t, rope_t, torch.from_numpy(slots).cuda(), cache, ks)
    got = cache.cpu().numpy().reshape(128, 576)[:, :512]
    empty = np.full((2, 64, 576), 0x7F, dtype=np.uint8)
    ref = O.cache_write(empty, latent, rope, slots, 64, F8, scale).reshape(128, 576)[:, :512]
    x = O.bf16_bits_to_f64(latent)
    nan_in = np.isnan(x)
    # NaN inputs: any NaN code is a correct encoding; everything else must match bit for bit
    assert np.isnan(fp8_e4m3.decode(got[nan_in])).all()
    assert np.array_equal(got[~nan_in], ref[~nan_in])


def test_cache_write_reports_out_of_range_slots():
    case = synth.make_case(B=1, s_q=1, H=1, page_size=64, seq_lens=[10], seed=22)
    g = GpuCase(case, build_cache=False)
    g.cache = g.empty_cache()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.from_numpy(case.slot_mapping.copy()).cuda()
    slots[3] = case.num_pages * case.page_size         # one past the pool
    api.cache_write(torch.from_numpy(case.latent_bits.view(np.int16)).view(torch.bfloat16).cuda(),
                    torch.from_numpy(case.rope_bits.view(np.int16)).view(torch.bfloat16).cuda(),
                    slots, g.cache, None, err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x10


# ---------------------------------------------------------------- decode, small
SMALL = [
    # B, s_q, H, P, lens, kv, causal
    (2, 1, 16, 64, [100, 257], BF, True),            # config 1 shape
    (1, 1, 16, 64, [1], BF, True),                   # a single key
    (3, 1, 16, 64, [127, 128, 129], BF, True),       # tile edges
    (2, 1, 16, 128, [63, 64], BF, True),
    (4, 1, 16, 64, [5000, 17, 640, 2049], BF, True), # several splits, ragged tail
    (2, 1, 128, 128, [300, 1000], BF, True),         # two row groups of 64
    (2, 1, 32, 64, [200, 129], BF, True),
    (2, 1, 20, 64, [77, 333], BF, True),             # a ragged row group
    (2, 1, 1, 64, [90, 700], BF, True),
    (2, 4, 128, 64, [1000, 67], F8, True),           # multi-token causal, FP8
    (3, 4, 16, 64, [4, 5, 130], BF, True),           # s_q = seq_len
    (2, 2, 16, 128, [300, 129], BF, False),          # non-causal multi-token
    (2, 1, 16, 64, [100, 257], F8, True),
    (3, 1, 128, 128, [1500, 130, 2000], F8, True),
    (2, 1, 64, 64, [4096, 3000], F8, True),
    (2, 3, 16, 64, [3, 129], F8, True),
    # more than 64 rows, bf16 cache: CTA pairs, 128-row groups, 256-key super-tiles
    (2, 1, 128, 64, [1, 255], BF, True),             # a single key; one short of a super-tile
    (3, 1, 128, 64, [256, 257, 513], BF, True),      # super-tile edges
    (3, 1, 128, 128, [64, 65, 190], BF, True),       # 64-key block edges, ragged 16-key steps
    (2, 1, 128, 128, [77, 4000], BF, True),          # split across many pairs, 128-row combine
    (2, 2, 128, 64, [300, 70], BF, True),            # two row groups, causal
    (2, 1, 96, 64, [500, 129], BF, True),            # a partly filled row group
    (2, 1, 100, 64, [500, 129], BF, True),           # rows not a multiple of 8: Q by chunks
    (2, 2, 64, 64, [1000, 65], BF, True),            # 128 rows from s_q = 2
    (1, 4, 128, 64, [5000], BF, False),              # four row groups, non-causal, splits
    (2, 1, 8, 64, [700, 1300], BF, True),            # H = 8 (TP = 16 of 128 heads)
    (2, 1, 64, 64, [900, 2100], BF, True),           # H = 64 (TP = 2)
    (2, 1, 16, 256, [300, 1100], BF, True),          # page size 256
    (2, 1, 128, 256, [300, 1100], BF, True),
    # multi-token decode (causal within the new tokens) up to the 512-token decode threshold
    (2, 8, 16, 64, [200, 700], BF, True),            # 128 rows
    (2, 64, 16, 64, [64, 900], BF, True),            # 1024 rows, s_q = seq_len for one sequence
    (1, 512, 16, 64, [1000], BF, True),              # 8192 rows, 64 row groups
    (2, 16, 128, 64, [300, 2000], BF, True),         # 2048 rows
    (2, 8, 16, 64, [200, 700], F8, True),            # FP8, two 64-row groups
    (2, 32, 64, 128, [40, 600], F8, True),           # FP8, 2048 rows
    # pages smaller than a 64-key block (boxes of gcd(P, 64) rows, several pages per block)
    (2, 1, 16, 16, [100, 257], BF, True),
    (3, 1, 16, 8, [1, 9, 300], BF, True),
    (2, 1, 32, 24, [200, 129], BF, True),            # P = 24: 8-row boxes
    (2, 1, 16, 1024, [300, 2000], BF, True),         # the largest page
    (2, 1, 16, 32, [100, 257], F8, True),
    (2, 1, 16, 48, [95, 700], F8, True),             # P = 48: 16-row boxes
    (2, 1, 64, 16, [500, 129], F8, True),
    (2, 4, 128, 32, [1000, 67], F8, True),
    (3, 1, 128, 16, [1, 255, 513], BF, True),        # CTA pairs
    (2, 1, 128, 8, [77, 1000], BF, True),
    (2, 1, 128, 48, [300, 70], BF, True),
    # more than 64 rows, FP8 cache: CTA pairs reading E4M3 directly (32-key MMA steps)
    (2, 1, 128, 64, [1, 255], F8, True),             # a single key; one short of a super-tile
    (3, 1, 128, 64, [256, 257, 513], F8, True),      # super-tile edges
    (3, 1, 128, 128, [64, 65, 190], F8, True),       # block edges, ragged 32-key steps
    (4, 1, 128, 128, [32, 33, 95, 96], F8, True),    # 32-key step edges
    (2, 1, 100, 64, [500, 129], F8, True),           # rows not a multiple of 8: Q by chunks
    # FP8 with 16 or 32 rows: E4M3 MMAs on whole-row key stages
    (1, 1, 16, 64, [1], F8, True),                   # a single key
    (3, 1, 16, 64, [127, 128, 129], F8, True),       # tile edges
    (4, 1, 16, 128, [32, 33, 95, 96], F8, True),     # 32-key step edges
    (4, 1, 16, 64, [5000, 17, 640, 2049], F8, True), # several splits, ragged tail
    (3, 1, 16, 8, [1, 9, 300], F8, True),            # 8-row pages
    (2, 1, 32, 64, [200, 129], F8, True),            # 32 rows
    (2, 1, 20, 64, [77, 333], F8, True),             # a ragged row group
    (2, 2, 16, 64, [300, 129], F8, False),           # 32 rows from s_q = 2, non-causal
    (2, 4, 4, 64, [700, 4], F8, True),               # 16 rows from s_q = 4, causal
    (3, 1, 32, 16, [1, 95, 300], F8, True),          # 16-row pages, 32 rows
    (4, 1, 16, 64, [95, 96, 97, 191], F8, True),     # 32-key step edges inside a tile
    (4, 1, 32, 128, [192, 193, 287, 288], F8, True), # the same, 32 rows
    (3, 1, 16, 96, [250, 1000, 97], F8, True),       # P = 96: 32-row boxes
    (2, 1, 16, 24, [300, 95], F8, True),             # P = 24: 8-row boxes
    (2, 3, 8, 64, [96, 1000], F8, True),             # 24 rows from s_q = 3, causal
    (2, 2, 64, 64, [1000, 65], F8, True),            # 128 rows from s_q = 2
    (3, 1, 128, 16, [1, 255, 513], F8, True),        # pages smaller than a block
    (2, 1, 128, 24, [77, 1000], F8, True),
]


@pytest.mark.parametrize("B,s_q,H,P,lens,kv,causal", SMALL)
def test_decode_matches_oracle_small(B, s_q, H, P, lens, kv, causal):
    case = synth.make_case(B=B, s_q=s_q, H=H, page_size=P, seq_lens=lens, seed=31 + B + H,
                           kv_dtype=kv, causal=causal)
    g = GpuCase(case)
    out, lse = g.decode()
    torch.cuda.synchronize()
    st, bits = api.decode_check(g.workspace)
    assert st == 0 and bits == 0
    ro, rl = oracle_decode(case, g.cache_numpy())
    compare(case, out, lse, ro, rl)


@pytest.mark.parametrize("kv", [BF, F8])
def test_pair_units_whose_odd_half_is_past_the_end_never_stall(kv):
    """CTA pairs: with 16 row groups over two sequences, pairs take a one-tile unit and then
    a unit whose second super-tile holds keys only in the even CTA's half. Every key slot
    needs bytes from both CTAs, so the odd CTA's producer stays in step with the slot's
    releases; before that, one run in ~14 stalled until the wait bound. Repeated calls must
    all succeed and give bit-identical results equal to the oracle's."""
    case = synth.make_case(B=2, s_q=16, H=128, page_size=64, seq_lens=[300, 2000], seed=31 + 2 + 128,
                           kv_dtype=kv, causal=True)
    g = GpuCase(case)
    out0, lse0 = [t.clone() for t in g.decode()]
    assert api.decode_check(g.workspace) == (0, 0)
    ro, rl = oracle_decode(case, g.cache_numpy())
    compare(case, out0, lse0, ro, rl)
    for _ in range(24):
        out, lse = g.decode()
        assert api.decode_check(g.workspace) == (0, 0)
        assert torch.equal(out, out0) and torch.equal(lse, lse0)


def test_config1_tiny_full():
    case = synth.make_config(1)
    g = GpuCase(case)
    out, lse = g.decode()
    ro, rl = oracle_decode(case, g.cache_numpy())
    compare(case, out, lse, ro, rl)


# ---------------------------------------------------------------- properties
def test_poisoned_unused_pages_and_tails_do_not_change_the_output():
    case = synth.make_case(B=3, s_q=2, H=16, page_size=64, seq_lens=[70, 129, 500], seed=41)
    g = GpuCase(case)
    out0, lse0 = [t.clone() for t in g.decode()]
    # replace every NaN (never-written) value with a large finite one
    c = g.cache.view(torch.int16)
    c[c == synth.BF16_NAN_BITS] = 0x4700       # bf16 32768.0
    out1, lse1 = g.decode()
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    assert torch.isfinite(out0.float()).all()


def test_page_permutation_is_invisible():
    case = synth.make_case(B=2, s_q=1, H=16, page_size=64, seq_lens=[400, 900], seed=42)
    g = GpuCase(case)
    out0, lse0 = [t.clone() for t in g.decode()]
    perm = torch.from_numpy(np.random.default_rng(5).permutation(case.num_pages)).cuda()
    new_cache = torch.empty_like(g.cache)
    new_cache[perm] = g.cache
    g.cache = new_cache
    g.block_table = perm[g.block_table.long()].int()
    out1, lse1 = g.decode()
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_garbage_workspace_and_outputs_are_fine():
    case = synth.make_case(B=4, s_q=1, H=16, page_size=64, seq_lens=[3000, 10, 700, 2500], seed=43)
    g = GpuCase(case)
    out0, lse0 = [t.clone() for t in g.decode()]
    g.workspace.fill_(0xFF)
    out = torch.full_like(out0, float("nan"))
    lse = torch.full_like(lse0, float("nan"))
    out1, lse1 = g.decode(out=out, lse=lse)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_repeated_calls_are_deterministic():
    case = synth.make_case(B=8, s_q=1, H=128, page_size=128, seq_lens=(100, 3000), seed=44, kv_dtype=F8)
    g = GpuCase(case)
    a = [t.clone() for t in g.decode()]
    b = g.decode()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_profile_window_times_the_decode_kernels_and_changes_nothing():
    """Events around the decode launch (a timing window of two calls) leave the results
    bit-identical; each window counts its launches and stops after max_launches."""
    case = synth.make_case(B=4, s_q=1, H=16, page_size=64, seq_lens=[3000, 10, 700, 2500], seed=46)
    g = GpuCase(case)
    out0, lse0 = [t.clone() for t in g.decode()]
    api.profile_begin(2)
    for _ in range(3):
        out1, lse1 = g.decode()
    ms, n = api.profile_end()
    assert n == 2 and 0.0 < ms < 1000.0
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    assert api.profile_end() == (0.0, 0)          # the window is closed


@pytest.mark.parametrize("H,P,kv,entry", [
    (16, 64, BF, (1, 2)), (16, 64, F8, (1, 2)), (128, 64, BF, (1, 2)), (64, 64, F8, (1, 2)),
    (16, 16, BF, (1, 9)), (16, 16, F8, (1, 9)), (128, 16, BF, (1, 9)),   # not a block's first page
])
def test_out_of_range_block_table_entry_is_reported_not_faulted(H, P, kv, entry):
    case = synth.make_case(B=2, s_q=1, H=H, page_size=P, seq_lens=[100, 200], seed=45, kv_dtype=kv)
    g = GpuCase(case)
    g.block_table[entry] = case.num_pages + 7
    g.decode()
    st, bits = api.decode_check(g.workspace)
    assert st == -6
    assert bits & 0x1


def test_fp8_query_beyond_the_float16_range_is_reported():
    """With an FP8 cache and 33-64 rows the MMAs run in fp16, so q is converted bf16 -> fp16;
    a query value above the fp16 range is flagged in the device error word
    (MLA_DEVERR_Q_RANGE) rather than silently saturated, and a clean call afterwards
    reports nothing."""
    case = synth.make_case(B=2, s_q=1, H=64, page_size=64, seq_lens=[100, 200], seed=47, kv_dtype=F8)
    g = GpuCase(case)
    q0 = g.q.clone()
    g.q[1, 0, 5, 17] = 1.0e5                       # a bf16 value, above 65504
    g.decode()
    st, bits = api.decode_check(g.workspace)
    assert st == -6 and bits & 0x4
    g.q = q0
    out, lse = g.decode()
    assert api.decode_check(g.workspace) == (0, 0)
    ro, rl = oracle_decode(case, g.cache_numpy())
    compare(case, out, lse, ro, rl)


def test_fp8_pairs_take_any_bf16_query_magnitude():
    """With an FP8 cache and more than 64 rows, each unit's q rows are scaled per row by a
    power of two before they are split into two E4M3 terms, so rows of very different
    magnitude (here 1e30, 1e-30, 3e38 and an all-zero row) decode like any other: no error
    bit, and the oracle's result within the FP8 tolerance."""
    case = synth.make_case(B=2, s_q=1, H=128, page_size=64, seq_lens=[700, 300], seed=49, kv_dtype=F8)
    q = torch.from_numpy(case.q_bits.view(np.int16).copy()).view(torch.bfloat16).float()
    q[0, 0, 3, :] *= 1.0e30
    q[0, 0, 77, :] *= 1.0e-30
    q[1, 0, 5, :] = 0.0
    q[1, 0, 9, :] = 0.0
    q[1, 0, 9, 100] = 3.0e38
    q[1, 0, 9, 101] = -1.0e-38
    case.q_bits[...] = q.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    g = GpuCase(case)
    out, lse = g.decode()
    assert api.decode_check(g.workspace) == (0, 0)
    ro, rl = oracle_decode(case, g.cache_numpy())
    # the output contract on every row; the LSE of rows scaled by 1e30 or 3e38 is itself of
    # that size, where one float32 step is ~1e23 to ~1e30: those get a relative bound
    lg = lse.cpu().numpy().astype(np.float64)
    big = np.abs(rl) > 1.0e6
    assert big.sum() == 2
    assert (np.abs(lg - rl)[big] <= 1.0e-6 * np.abs(rl[big])).all()
    compare(case, out, lse, ro, rl, rows=np.argwhere(~big))
    og = out.float().cpu().numpy().astype(np.float64)
    assert (np.abs(og - ro)[big] <= 2.0e-2).all()


@pytest.mark.parametrize("H", [16, 32])
def test_fp8_16_and_32_rows_take_any_bf16_query_magnitude(H):
    """With an FP8 cache and up to 32 rows the keys stay E4M3 in the MMAs too: each unit's q
    rows are scaled per row by a power of two and split into two E4M3 terms, so rows of very
    different magnitude (1e30, 1e-30, 3e38 with a tiny neighbour, all zero) decode with no
    error bit and within the FP8 tolerance of the oracle."""
    case = synth.make_case(B=2, s_q=1, H=H, page_size=64, seq_lens=[700, 300], seed=53 + H, kv_dtype=F8)
    q = torch.from_numpy(case.q_bits.view(np.int16).copy()).view(torch.bfloat16).float()
    q[0, 0, 3, :] *= 1.0e30
    q[0, 0, 7, :] *= 1.0e-30
    q[1, 0, 5, :] = 0.0
    q[1, 0, 9, :] = 0.0
    q[1, 0, 9, 100] = 3.0e38
    q[1, 0, 9, 101] = -1.0e-38
    case.q_bits[...] = q.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    g = GpuCase(case)
    out, lse = g.decode()
    assert api.decode_check(g.workspace) == (0, 0)
    ro, rl = oracle_decode(case, g.cache_numpy())
    lg = lse.cpu().numpy().astype(np.float64)
    big = np.abs(rl) > 1.0e6
    assert big.sum() == 2
    assert (np.abs(lg - rl)[big] <= 1.0e-6 * np.abs(rl[big])).all()
    compare(case, out, lse, ro, rl, rows=np.argwhere(~big))
    og = out.float().cpu().numpy().astype(np.float64)
    assert (np.abs(og - ro)[big] <= 2.0e-2).all()


@pytest.mark.parametrize("H,kv", [(16, BF), (16, F8), (128, BF), (128, F8)])
def test_a_stalled_pipeline_times_out_and_the_next_call_is_clean(H, kv):
    """Failure detection: with the wait bound shortened to 20 ms and the first softmax wait
    of every CTA made to wait on a barrier nothing arrives on, the call reports
    MLA_ERR_TIMEOUT (no fault, no hang); the kernel drained its copies and MMAs, so the
    next normal call on the same stream gives the oracle's result."""
    case = synth.make_case(B=3, s_q=1, H=H, page_size=64, seq_lens=[300, 2000, 70], seed=48, kv_dtype=kv)
    g = GpuCase(case)
    try:
        api.test_set_hooks(wait_limit_ns=20_000_000, stall=True)
        g.decode()
        st, bits = api.decode_check(g.workspace)
    finally:
        api.test_set_hooks(0, False)
    assert st == -5 and bits & 0x8
    out, lse = g.decode()
    assert api.decode_check(g.workspace) == (0, 0)
    ro, rl = oracle_decode(case, g.cache_numpy())
    compare(case, out, lse, ro, rl)


def test_bad_arguments_launch_nothing():
    case = synth.make_case(B=1, s_q=1, H=16, page_size=64, seq_lens=[10], seed=46)
    g = GpuCase(case)
    with pytest.raises(api.MLAError) as e:
        api.decode(g.q, g.cache, g.block_table, g.seq_lens, 0.1, max_seq_len=10,
                   workspace=g.workspace[:100])
    assert e.value.status == -3


# ----------------------------------------------------------- the longest sequence
@pytest.mark.parametrize("H,P,kv", [(16, 64, BF), (128, 128, F8)])
def test_the_longest_sequence_matches_the_oracle(H, P, kv):
    """A sequence of 2^20 keys (the largest max_seq_len the library takes) beside a short
    one: every row against the float64 oracle. The long stream is cut over every worker and
    merged by the combine kernel."""
    case = synth.make_case(B=2, s_q=1, H=H, page_size=P, seq_lens=[1 << 20, 300], seed=97 + H,
                           kv_dtype=kv)
    g = GpuCase(case)
    out, lse = g.decode()
    torch.cuda.synchronize()
    st, bits = api.decode_check(g.workspace)
    assert st == 0 and bits == 0
    ro, rl = oracle_decode(case, g.cache_numpy())
    compare(case, out, lse, ro, rl)


# ---------------------------------------------------------------- full-size configs
FULL = [(2, None, None), (3, None, None), (4, BF, None), (4, F8, None), (5, None, 1), (5, None, 4)]


@pytest.mark.parametrize("cfg,kv,s_q", FULL)
def test_full_size_configs_every_row(cfg, kv, s_q):
    """Each full-size workload, every output element and LSE against the float64 oracle (the
    oracle walks each sequence's pages once; seconds per workload on the host cores)."""
    case = synth.make_config(cfg, kv_dtype=kv, s_q=s_q)
    g = GpuCase(case)
    out, lse = g.decode()
    torch.cuda.synchronize()
    st, bits = api.decode_check(g.workspace)
    assert st == 0 and bits == 0
    cache = g.cache_numpy()
    if cfg == 3:
        ref_cache = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits,
                                  case.slot_mapping, case.page_size, case.kv_dtype, case.kv_scale)
        assert np.array_equal(cache, ref_cache)        # bit-exact FP8 write at full size
    ro, rl = oracle_decode(case, cache)
    compare(case, out, lse, ro, rl)
