"""Concurrent host threads: the library's per-device launch set-up (kernel
attributes, occupancy queries, SM counts, the device error word's address)
is filled once under a lock, so first calls made at the same time from
several threads, each on its own stream, give the same bytes as the same
calls made one after another.  Runs in a child process so that every cache
starts empty."""
import os
import subprocess
import sys
import textwrap

import pytest

from tests._util import need_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys, threading
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    from fp4_fp8_quantization_gb300 import moeq, synth
    torch.cuda.set_device(0)
    dev = "cuda"
    E, N, K = 6, 512, 1024
    counts = np.array([0, 1, 127, 129, 260, 3])
    ro = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    ids = np.array([4, 0, 2, 5, 1, 3], np.int32)
    so = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.uint32)
    T, rows = int(ro[-1]), int(so[-1])
    u32 = lambda x: torch.from_numpy(np.asarray(x, np.uint32).view(np.int32)).to(dev)
    x = synth.bf16_normal((T, K), 1.0, seed=3, device=dev)
    b = synth.random_fp4_packed((E, N, K // 2), seed=4, device=dev)
    bsf = synth.random_bytes(E * moeq.sf_bytes(N, K // 16), 0x18, 0x28, seed=5, device=dev)
    es = synth.uniform((E,), 0.5, 2.0, seed=6, device=dev)
    tk = torch.from_numpy(synth.topk_ids(512, 4, 64, seed=7)).to(dev)
    lg = synth.random_bytes(3 * 200 * 40, 0, 255, seed=8, device=dev).view(3, 200, 40)
    ro_d, so_d, ids_d = u32(ro), u32(so), torch.from_numpy(ids).to(dev)
    torch.cuda.synchronize()

    def work(stream):
        with torch.cuda.stream(stream):
            ts = torch.empty(E, device=dev)
            moeq.grouped_amax_scale(x, ro_d, ids_d, ts, E, stream=stream)
            a = torch.zeros((T, K // 2), dtype=torch.uint8, device=dev)
            asf = torch.zeros(moeq.sf_bytes(rows, K // 16), dtype=torch.uint8, device=dev)
            moeq.grouped_quantize("nvfp4", x, a, asf, ro_d, so_d, ids_d, ts, E, rows,
                                  stream=stream)
            y = torch.zeros((T, N), dtype=torch.bfloat16, device=dev)
            moeq.grouped_matmul_blockscaled("nvfp4", y, a, asf, b, bsf, es, ro_d, so_d, ids_d,
                                            N, K, rows, stream=stream)
            r_ro = torch.zeros(65, dtype=torch.int32, device=dev)
            r_ids = torch.zeros(64, dtype=torch.int32, device=dev)
            r_src = torch.zeros(tk.numel(), dtype=torch.int32, device=dev)
            moeq.route_topk(tk, r_ro, r_ids, r_src, stream=stream)
            t = torch.zeros(3 * moeq.sf_bytes(200, 40), dtype=torch.uint8, device=dev)
            moeq.sf_swizzle(t, lg, stream=stream)
        stream.synchronize()
        return [v.cpu() for v in (ts, a, asf, y, r_ro, r_src, t)]

    results = [None] * 8
    streams = [torch.cuda.Stream() for _ in range(8)]
    start = threading.Barrier(8)

    def run(i):
        start.wait()
        results[i] = work(streams[i])

    threads = [threading.Thread(target=run, args=(i,)) for i in range(8)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    ref = work(torch.cuda.Stream())
    for r in results:
        assert r is not None
        for got, want in zip(r, ref):
            assert torch.equal(got.view(torch.uint8), want.view(torch.uint8))
    assert moeq.get_device_error() == 0
    print("threads ok")
""")


def test_first_calls_from_eight_threads():
    need_gpu()
    code = "ROOT = %r\n" % ROOT + CHILD
    env = dict(os.environ)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600,
                       env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "threads ok" in r.stdout
