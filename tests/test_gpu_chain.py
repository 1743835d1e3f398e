"""Chained GEMM E = round(A.B1).B2 with the intermediate kept in tensor memory
as the second product's A operand, against the float64 oracle's
``gemm_chain`` (two oracle products around a round-to-nearest-even 16-bit
intermediate)."""
import numpy as np
import pytest
import torch

from gpu_helpers import OUT, U_OUT

pytestmark = pytest.mark.gpu

TAU = 2e-3
IN = {"f16": (0, torch.float16), "bf16": (1, torch.bfloat16)}   # tcg_input
ORACLE = {"f16": 1, "bf16": 2}
ULP = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7}   # spacing of 16-bit numbers, relative


@pytest.fixture(scope="module")
def tcg():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


def _inputs(dt, M, N1, N2, K, seed, integers=False):
    g = torch.Generator().manual_seed(seed)
    tdt = IN[dt][1]
    if integers:
        mk = lambda *s: torch.randint(-2, 3, s, generator=g).to(tdt)
    else:
        mk = lambda *s: torch.randn(*s, generator=g).to(tdt)
    return mk(M, K), mk(N1, K), mk(N2, N1)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _run(tcg, dt, A, B1, B2, out, lde=None, E=None):
    M, K = A.shape
    N1, N2 = B1.shape[0], B2.shape[0]
    lde = lde or N2
    if E is None:
        E = torch.full((M, lde), float("nan"), dtype=OUT[out][1], device="cuda")
    tcg.gemm_chain(IN[dt][0], M, N1, N2, K, A.cuda(), K, B1.cuda(), K, B2.cuda(), N1, E, OUT[out][0], lde)
    assert tcg.check() == 0
    return E


def _check(oracle_mod, dt, A, B1, B2, E, out, rows):
    M, K = A.shape
    N1, N2 = B1.shape[0], B2.shape[0]
    ref, S2, C, S1 = oracle_mod.gemm_chain(M, N1, N2, K, _bits(A), _bits(B1), _bits(B2), ORACLE[dt], rows=rows)
    got = E[rows, :N2].double().cpu().numpy()
    assert np.all(np.isfinite(got))
    # the GPU's fp32 intermediate is within TAU*S1 of the exact one; rounding
    # both to 16 bits can differ by that plus one spacing of the type
    dC = TAU * S1 + ULP[dt] * (np.abs(C) + TAU * S1)
    bound = dC @ np.abs(B2.double().numpy()).T + TAU * S2
    bound = bound + U_OUT[out] * (np.abs(ref) + bound)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:5].tolist())


EXACT = [
    # dt, M, N1, N2, K   (integers in [-2, 2]: every step exact, E bit for bit)
    ("bf16", 128, 16, 128, 64),
    ("bf16", 300, 48, 520, 120),
    ("f16", 257, 256, 200, 48),
    ("bf16", 1000, 128, 1032, 72),
    ("f16", 64, 80, 384, 200),
    ("bf16", 520, 16, 200, 64),    # N1 = 16: single CTAs even with several row tiles
    ("bf16", 2100, 128, 200, 64),  # B shared by CTA pairs; odd row-tile count: the last pair's second CTA idles
]


@pytest.mark.parametrize("dt,M,N1,N2,K", EXACT)
def test_chain_exact_on_small_integers(tcg, oracle_mod, dt, M, N1, N2, K):
    A, B1, B2 = _inputs(dt, M, N1, N2, K, seed=M + N1, integers=True)
    E = _run(tcg, dt, A, B1, B2, "f32")
    ref, _, _, _ = oracle_mod.gemm_chain(M, N1, N2, K, _bits(A), _bits(B1), _bits(B2), ORACLE[dt])
    assert np.array_equal(E.double().cpu().numpy(), ref)


RANDOM = [
    # dt, M, N1, N2, K, out
    ("bf16", 300, 64, 520, 256, "bf16"),
    ("bf16", 2048, 256, 1024, 512, "f32"),
    ("f16", 1000, 112, 2000, 1000, "f16"),
    ("bf16", 256, 256, 4000, 4096, "bf16"),     # 2 row tiles: E tiles split over many units
    ("bf16", 152 * 128 * 2 + 77, 128, 384, 512, "bf16"),  # more row tiles than SMs, ragged
    ("f16", 4000, 192, 700, 320, "f32"),     # CTA pairs, a B2 stage of one 64-column box after a full one
    ("f16", 2304, 256, 904, 320, "f16"),     # CTA pairs, f16 E, a ragged last E tile
]


@pytest.mark.parametrize("dt,M,N1,N2,K,out", RANDOM)
def test_chain_random_within_the_composed_bound(tcg, oracle_mod, dt, M, N1, N2, K, out):
    A, B1, B2 = _inputs(dt, M, N1, N2, K, seed=7 * M + K)
    E = _run(tcg, dt, A, B1, B2, out)
    rows = list(range(M)) if M <= 1024 else sorted({0, 1, 127, 128, 255, M // 2, M - 129, M - 2, M - 1} |
                                                    set(np.random.default_rng(M).integers(0, M, 16).tolist()))
    _check(oracle_mod, dt, A, B1, B2, E, out, rows)


def test_chain_matches_two_calls_through_a_16_bit_intermediate(tcg):
    # the same products through global memory: C = A.B1 stored as bf16, then
    # E = C.B2 (fp32 accumulation both times).  The MMAs see the same operands
    # in the same K order whether A comes from shared memory or from TMEM, so
    # the two agree bit for bit (measured); the bound below is what the
    # arithmetic alone guarantees
    dt, M, N1, N2, K = "bf16", 1024, 192, 640, 768
    A, B1, B2 = _inputs(dt, M, N1, N2, K, seed=11)
    E = _run(tcg, dt, A, B1, B2, "f32")
    C = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    tcg.gemm_bf16(M, N1, K, A.cuda(), 0, K, B1.cuda(), 0, K, C, 2, N1, 0)
    E2 = torch.empty((M, N2), dtype=torch.float32, device="cuda")
    tcg.gemm_bf16(M, N2, N1, C, 0, N1, B2.cuda(), 0, N1, E2, 0, N2, 0)
    assert tcg.check() == 0
    S = (C.double().abs() @ B2.cuda().double().abs().T)
    diff = (E.double() - E2.double()).abs()
    # an intermediate element may round the other way (one 16-bit spacing)
    assert bool((diff <= (ULP[dt] + 2 * TAU) * S + 1e-30).all())
    assert torch.equal(E, E2)


def test_chain_edges(tcg, oracle_mod):
    dt = "bf16"
    # K = 0: E is zeroed
    E = torch.full((50, 40), 3.0, dtype=torch.float32, device="cuda")
    z = torch.zeros(0, dtype=torch.bfloat16, device="cuda")
    B2 = torch.zeros((40, 16), dtype=torch.bfloat16, device="cuda")
    tcg.gemm_chain(1, 50, 16, 40, 0, z, 0, z, 0, B2, 16, E, 0, 40)
    assert tcg.check() == 0 and bool((E == 0).all())
    # M == 0 / N2 == 0: nothing happens, even with null pointers
    assert tcg.gemm_chain(1, 0, 16, 40, 64, None, 0, None, 0, None, 0, None, 0, 0, check=False) == 0
    assert tcg.gemm_chain(1, 50, 16, 0, 64, None, 0, None, 0, None, 0, None, 0, 0, check=False) == 0
    A, B1, B2 = _inputs(dt, 64, 32, 64, 64, seed=1)
    A, B1, B2 = A.cuda(), B1.cuda(), B2.cuda()
    E = torch.zeros((64, 72), dtype=torch.float32, device="cuda")
    for n1 in (0, 8, 24, 272):   # N1 a multiple of 16 in [16, 256]
        assert tcg.gemm_chain(1, 64, n1, 64, 64, A, 64, B1, 64, B2, 32, E, 0, 72, check=False) == tcg.ERR_INVALID
    # E's row stride must be a 16-byte multiple for its tile stores
    Ebf = torch.zeros((64, 68), dtype=torch.bfloat16, device="cuda")
    assert tcg.gemm_chain(1, 64, 32, 64, 64, A, 64, B1, 64, B2, 32, Ebf, 2, 67,
                          check=False) == tcg.ERR_ALIGNMENT
    # a padded E (lde > N2) leaves the padding alone
    E = torch.full((64, 72), 5.0, dtype=torch.float32, device="cuda")
    tcg.gemm_chain(1, 64, 32, 64, 64, A, 64, B1, 64, B2, 32, E, 0, 72)
    assert tcg.check() == 0 and bool((E[:, 64:] == 5.0).all())
    _check(oracle_mod, dt, A.cpu(), B1.cpu(), B2.cpu(), E, "f32", list(range(64)))


def test_chain_bench_workload_sampled_rows(tcg, oracle_mod):
    # the benchmark's chained workload at full size, its seeded inputs
    import synthetic as syn
    w = syn.WORKLOADS["chain_bf16_38912x256x4096"]
    x = syn.make_chain_inputs(w)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    A, B1, B2 = to(x["A"]), to(x["B1"]), to(x["B2"])
    E = _run(tcg, "bf16", A, B1, B2, w.out)
    M = w.M
    rows = sorted({0, 1, 31, 32, 127, 128, 255, 19456, M - 129, M - 2, M - 1} |
                  set(np.random.default_rng(3).integers(0, M, 12).tolist()))
    _check(oracle_mod, "bf16", A, B1, B2, E, w.out, rows)


@pytest.mark.parametrize("M,N1", [(700, 96), (2100, 128)])   # single CTAs; clusters of two sharing B
def test_chain_graph_capture_and_replay(tcg, M, N1):
    # one chained launch captured into a CUDA graph and replayed: identical
    # to the eager call every time
    dt, N2, K = "bf16", 600, 320
    A, B1, B2 = (t.cuda() for t in _inputs(dt, M, N1, N2, K, seed=21))
    eager = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tcg.gemm_chain(1, M, N1, N2, K, A, K, B1, K, B2, N1, eager, 2, N2, stream=s.cuda_stream)
        s.synchronize()
        assert tcg.check(s.cuda_stream) == 0
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            tcg.gemm_chain(1, M, N1, N2, K, A, K, B1, K, B2, N1, out, 2, N2, stream=s.cuda_stream)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert tcg.check() == 0
        assert torch.equal(out, eager)


def test_chain_cluster_rule(tcg):
    # clusters of two sharing B from 16 row tiles and N1 = 128 up; the parity
    # cases above cover both kinds of launch only if this rule holds
    A, B1, B2 = (t.cuda() for t in _inputs("bf16", 2100, 128, 200, 64, seed=5))
    E = torch.empty((2100, 200), dtype=torch.bfloat16, device="cuda")
    for n1, shared in ((128, True), (64, False)):
        tcg.gemm_chain(1, 2100, n1, 200, 64, A, 64, B1, 64, B2, 128, E, 2, 200)
        assert ("of 2 sharing B by multicast" in tcg.last_plan_string()) == shared, tcg.last_plan_string()
    tcg.gemm_chain(1, 1900, 128, 200, 64, A, 64, B1, 64, B2, 128, E, 2, 200)   # 15 row tiles
    assert "sharing B" not in tcg.last_plan_string()
    assert tcg.check() == 0


def test_chain_trace_records_entry_exit_and_units(tcg):
    # tcg_trace_next also covers the chained kernel: entry / exit stamps, the
    # cycle counter beside them, and the units each CTA's MMA warp computed
    A, B1, B2 = (t.cuda() for t in _inputs("bf16", 4096, 256, 1000, 256, seed=8))
    E = torch.empty((4096, 1000), dtype=torch.bfloat16, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros((sms, 10), dtype=torch.int64, device="cuda")
    tcg.trace_next(buf, sms)
    tcg.gemm_chain(1, 4096, 256, 1000, 256, A, 256, B1, 256, B2, 256, E, 2, 1000)
    assert tcg.check() == 0
    tr = buf.cpu().numpy()
    ran = tr[:, 0] > 0
    assert ran.sum() >= 32   # 32 row tiles, and the E tiles split into groups over the rest
    assert (tr[ran, 6] > tr[ran, 0]).all() and (tr[ran, 9] > tr[ran, 8]).all()
    assert (tr[ran, 7] >= 1).all() and tr[ran, 7].sum() >= 32
    ghz = (tr[ran, 9] - tr[ran, 8]) / (tr[ran, 6] - tr[ran, 0])
    assert ((ghz > 0.3) & (ghz < 3.0)).all(), ghz
    # the request is consumed: the next call writes nothing
    buf.zero_()
    tcg.gemm_chain(1, 4096, 256, 1000, 256, A, 256, B1, 256, B2, 256, E, 2, 1000)
    assert tcg.check() == 0 and int(buf.abs().sum()) == 0


def test_chain_single_ctas_and_clusters_agree_bit_for_bit(tcg):
    # 1900 rows (15 row tiles: single CTAs) and 2100 rows (17: clusters of
    # two sharing B by multicast) run the same MMAs in the same order on the
    # first 1900 rows of A, so those rows of E are identical
    A, B1, B2 = (t.cuda() for t in _inputs("bf16", 2100, 256, 700, 512, seed=13))
    E = {}
    for M in (1900, 2100):
        E[M] = torch.full((M, 700), float("nan"), dtype=torch.float32, device="cuda")
        tcg.gemm_chain(1, M, 256, 700, 512, A, 512, B1, 512, B2, 256, E[M], 0, 700)
        assert tcg.check() == 0
        assert ("sharing B" in tcg.last_plan_string()) == (M == 2100), tcg.last_plan_string()
    assert torch.equal(E[1900], E[2100][:1900])
