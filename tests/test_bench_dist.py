"""The multi-process timing logic of bench.py (barrier, max and sum over ranks), run as
two gloo ranks on CPU. The data path has no collective: ranks are independent replicas."""
import os
import socket
import subprocess
import sys
import textwrap

from conftest import ROOT

CHILD = textwrap.dedent("""
    import os, sys, json
    sys.path.insert(0, {root!r})
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo")
    r, lr, w = bench.dist_env()
    bench.barrier(w)
    mx = bench.max_over_ranks(float(10 + r), w)
    sm = bench.sum_over_ranks(float(1 + r), w)
    print(json.dumps({{"rank": r, "world": w, "max": mx, "sum": sm}}), flush=True)
    dist.destroy_process_group()
""")


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_gloo_ranks_agree_on_max_and_sum(tmp_path):
    script = tmp_path / "child.py"
    script.write_text(CHILD.format(root=ROOT))
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    import json
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o, _ in outs), key=lambda d: d["rank"])
    assert [d["world"] for d in res] == [2, 2]
    assert all(d["max"] == 11.0 for d in res)
    assert all(d["sum"] == 3.0 for d in res)


def test_kernel_source_hash_ignores_comments_only():
    """The DRAM-traffic table is keyed by a hash of the kernel code without its comments:
    an edit of a comment keeps the key, any change of code (or a string) changes it."""
    sys.path.insert(0, str(ROOT))
    import bench
    src = 'int a = 1; // one\n/* block\n comment */ const char* s = "x // y";\n'
    same = 'int a = 1;   // the value one\nconst char* s = "x // y"; /* other */\n'
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(src.replace("a = 1", "a = 2"))
    assert bench._code_only(src) != bench._code_only(src.replace('"x // y"', '"x /* y"'))
    assert len(bench.kernel_source_hash()) == 16
