"""Host-side logic of bench.py on the CPU: sharded timing over ranks (gloo, 2 ranks),
FLOP accounting and the reference-arm JSON contract."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    ws, r = bench.init_dist("gloo")
    t = bench.max_over_ranks(10.0 + 5.0 * rank)
    bench.barrier()
    from scaled_dot_product_tcgen05_gb300 import workloads as W
    wl = bench.shard_workload(W.standard_workloads()["long64k_causal"], r)
    q.put((r, ws, t, wl.base_seed, (wl.B, wl.H, wl.Sq, wl.D)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[:3] for g in got] == [(0, 2, 15.0), (1, 2, 15.0)]
    # each rank processes its own shard: same shapes, distinct seeded inputs
    assert got[0][4] == got[1][4] and got[0][3] != got[1][3]


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5


def test_workload_info_flops_and_bytes():
    from scaled_dot_product_tcgen05_gb300 import workloads as W
    wl = W.standard_workloads()["long64k_causal"]
    flops, nbytes, cfg = bench.workload_info(wl)
    assert flops == 4 * 32 * 65536 ** 2 * 128 / 2
    assert nbytes == 65536 * 32 * 128 * 2 * 4 + 65536 * 32 * 4
    assert cfg["workload"] == "long64k_causal"


def test_reference_arm_json_contract():
    env = dict(os.environ, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_causal", "--steps", "1", "--warmup", "3",
                        "--ref-rows", "16"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, PYTHONPATH=ROOT, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_causal"], capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_workload_info_for_the_extension_workloads():
    from scaled_dot_product_tcgen05_gb300 import workloads as W
    wls = W.standard_workloads()
    # sliding window: the exact count of visible (query, key) pairs
    wl = wls["window128k_causal"]
    f, _, cfg = bench.workload_info(wl)
    S, Wn, G = 131072, 4096, 64
    pairs = sum(min(i + 1, Wn) for i in range(S))  # G <= W: global rows see i + 1 keys too
    assert f == 4.0 * 128 * 32 * pairs and cfg["window"] == [4095, 0] and cfg["global_q"] == G
    # decode: bytes = K and V caches + q + o + lse; flops = 4 D per visible pair
    wl = wls["decode32k_b16_q4"]
    f, nb, cfg = bench.workload_info(wl)
    assert nb == 16 * 32768 * 32 * 128 * 4 + 16 * 4 * 32 * 128 * 4 + 16 * 32 * 4 * 4
    assert f == 4.0 * 128 * 16 * 32 * sum(32768 - 4 + t + 1 for t in range(4))
    # backward: 2.5 x the forward convention; 8 tensors of bytes
    wl = wls["bwd16k_causal"]
    f, nb, cfg = bench.workload_info(wl)
    assert f == 2.5 * 4 * 32 * 16384 ** 2 * 128 / 2 and cfg["backward"]
    assert nb == 16384 * 32 * 128 * 2 * 8 + 16384 * 32 * 4
    # fp8: the forward's flops, 1-byte inputs
    wl = wls["fp8_long64k_causal"]
    f, nb, cfg = bench.workload_info(wl)
    assert f == 4 * 32 * 65536 ** 2 * 128 / 2
    assert nb == 65536 * 32 * 128 * 5 + 65536 * 32 * 4 and cfg["fp8"].startswith("e4m3")


def test_visible_key_counts_matches_a_direct_count():
    from scaled_dot_product_tcgen05_gb300 import workloads as W
    import numpy as np
    for Sq, Sk, causal, win, g in [(9, 9, True, (2, 0), 0), (7, 11, False, (1, 3), 2),
                                   (10, 10, False, (-1, -1), 0), (6, 6, True, (-1, -1), 0)]:
        got = W.visible_key_counts(Sq, Sk, causal, win, g)
        want = []
        for i in range(Sq):
            n = 0
            for j in range(Sk):
                ok = True
                if i >= g:
                    ok = (win[0] < 0 or j >= i - win[0]) and (win[1] < 0 or j <= i + win[1])
                if causal and j > i:
                    ok = False
                n += ok
            want.append(n)
        assert np.array_equal(got, np.array(want))


def test_shards_keep_shapes_and_draw_their_own_inputs():
    from scaled_dot_product_tcgen05_gb300 import workloads as W
    wl = W.standard_workloads()["bwd16k_causal"]
    shards = [bench.shard_workload(wl, r) for r in range(8)]
    assert shards[0] is wl
    assert len({s.base_seed for s in shards}) == 8
    assert all((s.B, s.H, s.Sq, s.Sk, s.D, s.causal, s.backward) ==
               (wl.B, wl.H, wl.Sq, wl.Sk, wl.D, wl.causal, wl.backward) for s in shards)
    # no shard's seed collides with another workload family's
    others = {w.base_seed for n, w in W.standard_workloads().items() if w.wid != wl.wid}
    assert not ({s.base_seed for s in shards} & others)


def test_seed_selects_another_draw_of_the_same_workload():
    from scaled_dot_product_tcgen05_gb300 import workloads as W
    wl = W.standard_workloads()["long64k_causal"]
    assert bench.reseed_workload(wl, 0) is wl
    seeds = [bench.reseed_workload(wl, s) for s in range(10)]
    assert len({s.base_seed for s in seeds}) == 10
    assert all((s.B, s.H, s.Sq, s.D, s.causal) == (wl.B, wl.H, wl.Sq, wl.D, wl.causal)
               for s in seeds)
    # reseeded and sharded draws of every workload stay inside its family's seed block
    for w in W.standard_workloads().values():
        for s in range(10):
            for r in range(8):
                x = bench.shard_workload(bench.reseed_workload(w, s), r)
                assert x.base_seed // 1000 == w.wid
    with pytest.raises(SystemExit):
        bench.reseed_workload(wl, 10)


def test_l2_flush_only_for_steps_that_fit_in_l2():
    """Workloads whose step touches less than twice the L2 are flushed between timed
    steps (the 2K, 512 and tiny ones); the long, packed, window, decode and backward
    workloads are not."""
    l2 = bench.L2_BYTES
    assert bench.l2_flush_bytes(2 * l2) == 0
    assert bench.l2_flush_bytes(2 * l2 - 1) == 2 * l2
    assert bench.l2_flush_bytes(0) == 2 * l2
    wl = bench.W.standard_workloads()
    for name, flushed in [("mha2k_bf16_causal", True), ("mha512_causal", True), ("tiny_causal", True),
                          ("long64k_causal", False), ("varlen_causal", False),
                          ("window128k_causal", False), ("decode128k_q1", False)]:
        w = wl[name]
        _, nbytes, _ = bench.workload_info(w)  # inputs read and outputs written once
        assert (bench.l2_flush_bytes(int(nbytes)) > 0) == flushed, name


def test_committed_profiles_match_the_kernel_sources():
    """Every ncu summary under profiles/ names a benchmarked kernel and workload and
    records the digest of that kernel's sources; bench.py reports its DRAM traffic only
    while the digest matches, so a summary left behind by a kernel change shows here."""
    import re
    names = os.listdir(bench.PROFILE_DIR)
    assert names, "no profiles committed"
    wls = bench.W.standard_workloads()
    for name in names:
        assert name.endswith(".md"), name
        kernel = next((k for k in sorted(bench.KERNEL_SOURCES, key=len, reverse=True)
                       if name.startswith(k + "_")), None)
        assert kernel is not None, name
        workload = name[len(kernel) + 1:-3]
        assert workload in wls, name
        text = open(os.path.join(bench.PROFILE_DIR, name)).read()
        m = re.search(r"source_digest:\s*([0-9a-f]+)", text)
        assert m and m.group(1) == bench.source_digest(kernel), f"{name}: stale digest"
        assert bench.profiled_traffic(workload, kernel) > 0, name
