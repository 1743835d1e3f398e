"""Use from serving code: CUDA-graph capture and concurrent streams.

The calls are asynchronous on their stream and allocate only per-(device,
stream) workspaces on first use, so after one warm-up call on a stream they
can be captured into a CUDA graph and replayed; calls on different streams
use different workspaces and may run concurrently.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TAU, assert_parity, make_case, oracle_rows, to_device

pytestmark = pytest.mark.gpu

IN = {"f16": 0, "bf16": 1, "tf32": 2, "e4m3": 3}


@pytest.fixture(scope="module")
def tcg():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


def _enqueue(tcg, x, D, stream, split_k=0):
    w = x["w"]
    kw = {}
    if w.dtype == "e4m3":
        kw = dict(SFA=x["dSFA"], SFB=x["dSFB"])
    tcg.gemm(x["M"], x["N"], x["K"], IN[w.dtype], x["dA"], 0 if w.a_major == "k" else 1, x["lda"], x["dB"],
             0 if w.b_major == "k" else 1, x["ldb"], D, 2, x["N"], 0, split_k=split_k, stream=stream, **kw)


def _prepare(x):
    x["dA"], x["dB"] = to_device(x["A"]), to_device(x["B"])
    if x["w"].dtype == "e4m3":
        x["dSFA"], x["dSFB"] = to_device(x["SFA"]), to_device(x["SFB"])
    return x


def _check(oracle_mod, x, D, what):
    ref, S = oracle_rows(oracle_mod, x)
    assert_parity(D[:x["M"], :x["N"]].double().cpu().numpy(), ref, S, TAU["f32"], what, "bf16")


def test_graph_capture_and_replay(tcg, oracle_mod):
    # one pass per tile, stream-K (skinny), MXFP8 with plain scales (two
    # launches: scale rearrangement + GEMM)
    cases = [(_prepare(make_case("bf16", "k", "k", 300, 520, 256, seed=71)), 0),
             (_prepare(make_case("bf16", "k", "k", 16, 1000, 4096, seed=72)), -1),
             (_prepare(make_case("e4m3", "k", "k", 260, 460, 512, seed=73)), 0)]
    outs = [torch.full((x["M"], x["N"]), float("nan"), dtype=torch.bfloat16, device="cuda") for x, _ in cases]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for (x, sk), D in zip(cases, outs):  # warm-up: allocates this stream's workspaces
            _enqueue(tcg, x, D, s.cuda_stream, sk)
        s.synchronize()
        assert tcg.check(s.cuda_stream) == 0
        for D in outs:
            D.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for (x, sk), D in zip(cases, outs):
                _enqueue(tcg, x, D, s.cuda_stream, sk)
    for _ in range(3):
        for D in outs:
            D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert tcg.check() == 0
        for (x, _), D in zip(cases, outs):
            _check(oracle_mod, x, D, f"graph replay {x['w'].dtype} {x['M']}x{x['N']}x{x['K']}")


def test_concurrent_streams(tcg, oracle_mod):
    # the same problems on two streams at once; stream-K and MXFP8 use each
    # stream's own workspaces
    cases = [_prepare(make_case("bf16", "k", "k", 16, 1000, 4096, seed=81)),
             _prepare(make_case("e4m3", "k", "k", 300, 520, 256, seed=82))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[torch.full((x["M"], x["N"]), float("nan"), dtype=torch.bfloat16, device="cuda") for x in cases]
            for _ in streams]
    torch.cuda.synchronize()
    for rep in range(4):
        for st, row in zip(streams, outs):
            for x, D in zip(cases, row):
                _enqueue(tcg, x, D, st.cuda_stream, -1 if x["w"].dtype == "bf16" else 0)
    torch.cuda.synchronize()
    for st in streams:
        assert tcg.check(st.cuda_stream) == 0
    for row in outs:
        for x, D in zip(cases, row):
            _check(oracle_mod, x, D, f"stream {x['w'].dtype}")


def test_concurrent_host_threads(tcg, oracle_mod):
    # two host threads, each with its own stream, issue GEMMs at the same time
    # (the library's shared state is mutex-guarded; per-thread error strings)
    import threading
    cases = [_prepare(make_case("bf16", "k", "k", 16, 1000, 4096, seed=91)),
             _prepare(make_case("e4m3", "k", "k", 260, 460, 512, seed=92))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[torch.full((x["M"], x["N"]), float("nan"), dtype=torch.bfloat16, device="cuda") for x in cases]
            for _ in streams]
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            for rep in range(10):
                for x, D in zip(cases, outs[i]):
                    _enqueue(tcg, x, D, streams[i].cuda_stream, -1 if x["w"].dtype == "bf16" else 0)
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for st in streams:
        assert tcg.check(st.cuda_stream) == 0
    for row in outs:
        for x, D in zip(cases, row):
            _check(oracle_mod, x, D, f"thread {x['w'].dtype}")
