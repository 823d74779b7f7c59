"""The data-parallel replica driver, host side: every sequence is decoded by exactly one rank,
the ranks' token counts are balanced, every rank addresses only its own page pool, and a
rank's local decode (float64 oracle on its own cache and block table) equals the decode of
the whole batch for its sequences. The ranks run as two gloo processes; the only
collective is the test's own gather of what each rank saw."""
import json
import os
import socket
import subprocess
import sys
import textwrap

import numpy as np
import pytest

from conftest import ROOT
from mla_paged_decode_02_gb300 import replicas, synth
from oracle import mla_oracle as O


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_every_sequence_goes_to_one_rank_and_loads_balance(world):
    lens = np.random.default_rng(world).integers(1, 5000, size=37)
    parts = replicas.assign(lens, world)
    allidx = np.concatenate(parts)
    assert sorted(allidx.tolist()) == list(range(len(lens)))
    loads = [int(lens[p].sum()) for p in parts]
    assert max(loads) - min(loads) <= int(lens.max())


def test_a_shard_addresses_only_its_own_pool():
    lens = [100, 257, 4000, 64, 65, 1]
    for rank in range(2):
        s = replicas.shard(lens, 64, 2, rank, seed=3)
        for b, L in enumerate(s.seq_lens):
            pages = s.block_table[b, :-(-int(L) // 64)]
            assert pages.min() >= 0 and pages.max() < s.num_pages
        used = np.concatenate([s.block_table[b, :-(-int(L) // 64)] for b, L in enumerate(s.seq_lens)])
        assert len(np.unique(used)) == len(used)               # no page shared by two sequences


def local_oracle(case, world, rank):
    """The rank's decode on its own pool (float64 oracle), and the global decode's rows."""
    s = replicas.shard(case.seq_lens, case.page_size, world, rank, seed=5)
    rows, slots = replicas.local_token_rows(s, case.meta["tok_base"])
    shape = (s.num_pages, case.page_size, 576)
    empty = np.full(shape, synth.BF16_NAN_BITS, np.uint16) if case.kv_dtype == synth.KV_BF16 \
        else np.full(shape, synth.FP8_NAN_BYTE, np.uint8)
    cache = O.cache_write(empty, case.latent_bits[rows], case.rope_bits[rows], slots, case.page_size,
                          case.kv_dtype, case.kv_scale)
    out, lse = O.mla_decode(case.q_bits[s.seq_idx], cache, s.block_table, s.seq_lens, case.page_size,
                            case.softmax_scale, case.kv_dtype, case.kv_scale, case.causal)
    return s, out, lse


CHILD = textwrap.dedent("""
    import json, sys
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import numpy as np
    import torch.distributed as dist
    from mla_paged_decode_02_gb300 import synth
    from test_replicas import local_oracle
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    case = synth.make_case(B=5, s_q=2, H=4, page_size=64, seq_lens=[90, 700, 300, 1200, 65], seed=9,
                           kv_dtype={kv})
    s, out, lse = local_oracle(case, world, rank)
    res = {{"rank": rank, "seq_idx": s.seq_idx.tolist(), "tokens": int(s.seq_lens.sum()),
            "out": out.tolist(), "lse": lse.tolist()}}
    got = [None] * world
    dist.all_gather_object(got, res)          # the test's check only: the decode has no collective
    if rank == 0:
        print(json.dumps(got))
    dist.destroy_process_group()
""")


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8_E4M3])
def test_two_gloo_ranks_decode_the_batch_between_them(tmp_path, kv):
    script = tmp_path / "child.py"
    script.write_text(CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), kv=kv))
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=240) for p in procs]
    assert all(p.returncode == 0 for p in procs), [o[1][-2000:] for o in outs]
    got = json.loads(outs[0][0].strip().splitlines()[-1])
    case = synth.make_case(B=5, s_q=2, H=4, page_size=64, seq_lens=[90, 700, 300, 1200, 65], seed=9, kv_dtype=kv)
    cache = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits, case.slot_mapping,
                          case.page_size, kv, case.kv_scale)
    ref_out, ref_lse = O.mla_decode(case.q_bits, cache, case.block_table, case.seq_lens, case.page_size,
                                    case.softmax_scale, kv, case.kv_scale, case.causal)
    seen = []
    for r in got:
        idx = r["seq_idx"]
        seen += idx
        assert np.allclose(np.array(r["out"]), ref_out[idx], rtol=0, atol=1e-12)
        assert np.allclose(np.array(r["lse"]), ref_lse[idx], rtol=0, atol=1e-12)
    assert sorted(seen) == list(range(case.B))


@pytest.mark.gpu
@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8_E4M3])
def test_replicas_decode_their_shards_on_the_gpu(kv):
    """Each rank's Replica (its own pool, block table and cache written by mla_cache_write)
    decodes its sequences through the CUDA path; run here one rank after the other on one
    GPU (the ranks' kernels never wait on each other)."""
    import torch
    from gpu_harness import compare
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    case = synth.make_case(B=6, s_q=1, H=128, page_size=64, seq_lens=[90, 2700, 300, 1200, 65, 4000], seed=11,
                           kv_dtype=kv)
    cache = O.cache_write(case.empty_cache(), case.latent_bits, case.rope_bits, case.slot_mapping,
                          case.page_size, kv, case.kv_scale)
    ref_out, ref_lse = O.mla_decode(case.q_bits, cache, case.block_table, case.seq_lens, case.page_size,
                                    case.softmax_scale, kv, case.kv_scale, case.causal)
    for rank in range(2):
        s = replicas.shard(case.seq_lens, case.page_size, 2, rank, seed=7)
        rep = replicas.Replica(s, case.latent_bits, case.rope_bits, case.meta["tok_base"], kv, case.kv_scale, "cuda")
        out, lse = rep.decode(case.q_bits, case.softmax_scale, case.causal)
        torch.cuda.synchronize()
        local = synth.make_case(B=len(s.seq_idx), s_q=1, H=128, page_size=64, seq_lens=list(s.seq_lens), seed=0,
                                kv_dtype=kv)
        local.kv_dtype = kv
        compare(local, out, lse, ref_out[s.seq_idx], ref_lse[s.seq_idx])
