"""GPU parity tests: libgemm.so (through its C ABI) against the fp64 oracle.

Every case draws seeded inputs from the workload generators, runs the CUDA
path, and compares element by element with the oracle on the same host
values (tolerances in gpu_helpers).  Sizes span several tiles and a ragged
tail; the full-size workloads are checked on sampled entries.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import GuardedC, check_against_oracle, to_device_padded
from stage_software_pipelining_gb300 import build as gemm_build
from stage_software_pipelining_gb300 import gemm as G
from stage_software_pipelining_gb300.workloads import (BY_NAME, GEMM_BF16_BF16, GEMM_BF16_F32,
                                                       GEMM_F16_F32, GEMM_F32, OUT_DTYPE,
                                                       make_inputs)

pytestmark = pytest.mark.gpu

TC_DTYPES = [GEMM_F16_F32, GEMM_BF16_F32, GEMM_BF16_BF16]
BASE_FOR = {GEMM_F32: "fp32_256", GEMM_F16_F32: "fp16_2048", GEMM_BF16_F32: "bf16_8192_beta1",
            GEMM_BF16_BF16: "bf16_ragged_colB"}


@pytest.fixture(scope="module", autouse=True)
def library(gpu):
    gemm_build.build()
    G.load_library()
    G.debug_set(0, -1)
    yield
    G.debug_set(0, -1)


def workload(dtype, M, N, K, **kw):
    w = BY_NAME[BASE_FOR[dtype]].resized(M, N, K)
    return dataclasses.replace(w, **kw) if kw else w


def run_gpu(inp, stages, tile=0, alpha=None, beta=None, checked=True, guard=True):
    """Run the CUDA path on padded device copies; return (host C as float64, guard)."""
    w = inp.workload
    alpha = w.alpha if alpha is None else alpha
    beta = w.beta if beta is None else beta
    A = to_device_padded(inp.A)
    B = to_device_padded(inp.B, col_major=w.b_col_major)
    out_dt = OUT_DTYPE[w.dtype]
    init = inp.C0 if inp.C0 is not None else None
    gC = GuardedC(w.M, w.N, out_dt, init=init.cuda() if init is not None else None)
    if init is None:
        gC.view.fill_(float("nan") if beta == 0.0 else 0.0)
    G.gemm(A, B, gC.view, alpha, beta, stages=stages, tile=tile, checked=checked)
    torch.cuda.synchronize()
    if guard:
        gC.check()
    return gC.view.double().cpu().numpy(), gC


def oracle_full(inp, alpha=None, beta=None):
    w = inp.workload
    alpha = w.alpha if alpha is None else alpha
    beta = w.beta if beta is None else beta
    return oracle.gemm(inp.A, inp.B, inp.C0 if beta != 0.0 else None, alpha, beta)


# --------------------------------------------------------------------------- SIMT fp32
@pytest.mark.parametrize("stages", [1, 2, 3, 4])
def test_simt_fp32_256_matches_oracle(stages):
    inp = make_inputs(BY_NAME["fp32_256"])
    out, _ = run_gpu(inp, stages)
    ref, absb = oracle_full(inp)
    check_against_oracle(out, ref, absb, GEMM_F32, what=f"simt stages={stages}")


@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 15, 17), (129, 65, 33), (300, 200, 129),
                                   (128, 64, 16), (255, 127, 1)])
@pytest.mark.parametrize("stages", [1, 2])
def test_simt_ragged_shapes(shape, stages):
    M, N, K = shape
    inp = make_inputs(workload(GEMM_F32, M, N, K))
    out, _ = run_gpu(inp, stages)
    ref, absb = oracle_full(inp)
    check_against_oracle(out, ref, absb, GEMM_F32, what=f"simt {shape} s={stages}")


def test_simt_alpha_beta():
    w = workload(GEMM_F32, 200, 136, 72, alpha=-0.5, beta=2.0)
    inp = make_inputs(w)
    inp.C0 = torch.rand(200, 136, generator=torch.Generator().manual_seed(5)) * 2 - 1
    out, _ = run_gpu(inp, 2)
    ref, absb = oracle_full(inp)
    check_against_oracle(out, ref, absb, GEMM_F32, beta=2.0, C0=inp.C0, what="simt alpha/beta")


def test_simt_stage_invariance_bitwise():
    inp = make_inputs(workload(GEMM_F32, 333, 250, 190))
    outs = [run_gpu(inp, s)[0] for s in (1, 2, 3, 4)]
    for s, o in zip((2, 3, 4), outs[1:]):
        assert np.array_equal(o, outs[0]), f"SIMT stages={s} differs from stages=1"


def simt_split_plan(M, N, K):
    """The SIMT kernel's tail schedule, restated from its rule: 3 CTAs per SM
    make a wave; the tiles of a partial last wave are cut along K into
    min(8, wave // leftover, K tiles of 32 // 2) pieces when that is at
    least 2 (a piece spans at least 64 of K)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = -(-M // 128) * -(-N // 64)
    KT = -(-K // 32)
    W = 3 * sms
    R = T % W
    if R > 0:
        parts = min(8, W // R, KT // 2)
        if parts >= 2:
            return T - R, parts
    return T, 1


@pytest.mark.parametrize("shape", [(2176, 1792, 256), (2180, 1790, 250), (2048, 2048, 512)])
def test_simt_split_tail_matches_oracle_and_is_stage_invariant(shape):
    """Shapes whose last wave of 128 x 64 tiles is partial: those tiles run as
    K pieces combined through the workspace (also with ragged M, N, K and a
    K that leaves short pieces).  Every stage count gives the same bits, the
    bits match a second call, and the result matches the oracle."""
    M, N, K = shape
    dp, parts = simt_split_plan(M, N, K)
    assert parts >= 2, "the shape must exercise the split tail"
    assert G.plan(M, N, K, GEMM_F32, 2)["grid"] == dp + (-(-M // 128) * -(-N // 64) - dp) * parts
    inp = make_inputs(workload(GEMM_F32, M, N, K))
    outs = [run_gpu(inp, s)[0] for s in (1, 2, 3, 4)]
    again, _ = run_gpu(inp, 2)
    for s, o in zip((2, 3, 4), outs[1:]):
        assert np.array_equal(o, outs[0]), f"SIMT split tail: stages={s} differs from stages=1"
    assert np.array_equal(again, outs[1]), "a second call gives other bits"
    ref, absb = oracle_full(inp)
    check_against_oracle(outs[0], ref, absb, GEMM_F32, what=f"simt split tail {shape}")


def test_simt_split_tail_alpha_beta_and_streams():
    """beta != 0 is applied once, by the piece that finishes the tile; two
    streams at once use two workspaces."""
    M, N, K = 2176, 1792, 192
    assert simt_split_plan(M, N, K)[1] >= 2
    w = workload(GEMM_F32, M, N, K, alpha=-0.5, beta=2.0)
    inp = make_inputs(w)
    inp.C0 = torch.rand(M, N, generator=torch.Generator().manual_seed(8)) * 2 - 1
    A, B = inp.A.cuda(), inp.B.cuda()
    C1, C2 = inp.C0.cuda(), inp.C0.cuda()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        C1.copy_(inp.C0)
        C2.copy_(inp.C0)
        torch.cuda.synchronize()
        G.gemm(A, B, C1, w.alpha, w.beta, stages=2, stream=s1)
        G.gemm(A, B, C2, w.alpha, w.beta, stages=3, stream=s2)
        torch.cuda.synchronize()
        assert torch.equal(C1, C2)
    ref, absb = oracle_full(inp)
    check_against_oracle(C1.double().cpu().numpy(), ref, absb, GEMM_F32, beta=2.0, C0=inp.C0,
                         what="simt split tail alpha/beta")


@pytest.mark.parametrize("stages", [1, 2, 3, 4])
def test_simt_register_fragment_schemes_agree_bitwise(stages):
    """Double-buffered and single register fragments accumulate in the same
    order, so they give the same bits; both match the oracle."""
    inp = make_inputs(workload(GEMM_F32, 301, 198, 150))
    dbl, _ = run_gpu(inp, stages, tile=G.SIMT_FRAGMENTS_DOUBLE)
    single, _ = run_gpu(inp, stages, tile=G.SIMT_FRAGMENTS_SINGLE)
    assert np.array_equal(dbl, single)
    ref, absb = oracle_full(inp)
    check_against_oracle(dbl, ref, absb, GEMM_F32, what=f"simt fragments s={stages}")


# --------------------------------------------------------------------------- tensor cores
TILES = [G.TILE_128x128, G.TILE_128x256, G.TILE_256x256_2SM, G.TILE_256x512_2SM]
TILE_STAGES = {t: list(range(1, G.TILE_MAX_STAGES[t] + 1)) for t in TILES}


@pytest.mark.parametrize("dtype", TC_DTYPES)
@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("b_col_major", [False, True])
def test_tc_ragged_matches_oracle(dtype, tile, b_col_major):
    # several tiles with ragged M, N and K tails (for the 256 x 256 pair tile
    # the second tile row leaves the second CTA entirely out of range)
    w = workload(dtype, 300, 520, 200, b_col_major=b_col_major, beta=0.0)
    inp = make_inputs(w)
    out, _ = run_gpu(inp, 3, tile=tile)
    ref, absb = oracle_full(inp)
    check_against_oracle(out, ref, absb, dtype, what=f"tc dt={dtype} tile={tile} "
                                                      f"colB={b_col_major}")


@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 15, 17), (128, 256, 64), (129, 257, 65),
                                   (255, 129, 1000), (64, 1000, 8), (513, 384, 320)])
@pytest.mark.parametrize("b_col_major", [False, True])
def test_tc_shape_fuzz(shape, b_col_major):
    M, N, K = shape
    for dtype in (GEMM_BF16_F32, GEMM_F16_F32):
        inp = make_inputs(workload(dtype, M, N, K, b_col_major=b_col_major, beta=0.0))
        ref, absb = oracle_full(inp)
        for tile in (G.TILE_AUTO, G.TILE_128x256, G.TILE_256x256_2SM):
            out, _ = run_gpu(inp, 3, tile=tile)
            check_against_oracle(out, ref, absb, dtype, what=f"tc fuzz {shape} dt={dtype} "
                                                              f"tile={tile}")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("b_col_major", [False, True])
def test_tc_k_tails_across_the_atoms_of_a_stage(tile, b_col_major):
    """A stage holds K = 64 (one 128-byte swizzle row of 16-bit data): K ends
    inside a stage, exactly at a stage edge, and one or two stages past it,
    so that the last copy of a tile is partly past K (zero fill) and the ring
    wraps with 2 stages.  beta = 1 exercises the C box copies too."""
    for K in (8, 56, 64, 72, 120, 128, 136, 192, 200, 248, 256, 264):
        inp = make_inputs(workload(GEMM_BF16_F32, 200, 300, K, b_col_major=b_col_major, beta=1.0))
        out, _ = run_gpu(inp, 2, tile=tile)
        ref, absb = oracle_full(inp)
        check_against_oracle(out, ref, absb, GEMM_BF16_F32, beta=1.0, C0=inp.C0,
                             what=f"K tail K={K} tile={tile} colB={b_col_major}")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("dtype", TC_DTYPES)
def test_tc_stage_invariance_bitwise(tile, dtype):
    """The ring depth changes timing only: every stage count gives the same bits."""
    stages_list = TILE_STAGES[tile]
    w = workload(dtype, 384, 640, 520, beta=0.0)
    inp = make_inputs(w)
    outs = {s: run_gpu(inp, s, tile=tile)[0] for s in stages_list}
    ref, absb = oracle_full(inp)
    check_against_oracle(outs[stages_list[0]], ref, absb, dtype, what="tc invariance base")
    for s in stages_list[1:]:
        assert np.array_equal(outs[s], outs[stages_list[0]], equal_nan=True), \
            f"stages={s} differs from stages={stages_list[0]} (tile={tile})"


@pytest.mark.parametrize("alpha,beta", [(1.0, 1.0), (-0.5, 2.0), (2.0, -1.0), (0.25, 0.0)])
@pytest.mark.parametrize("dtype", TC_DTYPES)
@pytest.mark.parametrize("tile", [G.TILE_128x256, G.TILE_256x256_2SM])
def test_tc_alpha_beta(alpha, beta, dtype, tile):
    w = workload(dtype, 260, 300, 136, alpha=alpha, beta=beta)
    inp = make_inputs(w)
    if inp.C0 is None and beta != 0.0:
        gen = torch.Generator().manual_seed(99)
        inp.C0 = (torch.rand(260, 300, generator=gen) * 2 - 1).to(OUT_DTYPE[dtype])
    out, _ = run_gpu(inp, 2, tile=tile, alpha=alpha, beta=beta)
    ref, absb = oracle_full(inp, alpha, beta)
    check_against_oracle(out, ref, absb, dtype, beta=beta, C0=inp.C0,
                         what=f"alpha={alpha} beta={beta}")


@pytest.mark.parametrize("tile", TILES)
def test_beta_one_adds_c_with_one_fp32_rounding(tile):
    """With beta = 1 and fp32 C the epilogue adds alpha*acc into C at L2
    (tensor reduce): the result must be C0 + (the beta = 0 result) with one
    fp32 rounding, bit for bit, also for subnormal C0 and a ragged N edge."""
    M, N, K = 300, 1000, 264
    inp = make_inputs(workload(GEMM_BF16_F32, M, N, K, beta=1.0))
    A = to_device_padded(inp.A)
    B = to_device_padded(inp.B)
    C0 = inp.C0.cuda()
    C0[:7] *= 1e-39                                   # subnormal rows
    prod = torch.zeros(M, N, device="cuda")
    G.gemm(A, B, prod, 1.5, 0.0, stages=2, tile=tile, checked=True)
    C = C0.clone()
    G.gemm(A, B, C, 1.5, 1.0, stages=2, tile=tile, checked=True)
    assert torch.equal(C, C0 + prod)
    # A = 0: C0, subnormals included, comes back unchanged
    Cz = C0.clone()
    G.gemm(torch.zeros_like(A), B, Cz, 1.0, 1.0, stages=2, tile=tile, checked=True)
    assert torch.equal(Cz, C0)


@pytest.mark.parametrize("dtype", [GEMM_F32] + TC_DTYPES)
def test_beta_zero_does_not_read_c(dtype):
    inp = make_inputs(workload(dtype, 140, 136, 40, beta=0.0))
    out, _ = run_gpu(inp, 2)           # C is NaN-filled before the call
    assert np.isfinite(out).all()
    ref, absb = oracle_full(inp)
    check_against_oracle(out, ref, absb, dtype, what="beta=0 NaN C")


@pytest.mark.parametrize("dtype", [GEMM_F32, GEMM_BF16_F32, GEMM_BF16_BF16])
def test_k_zero_and_alpha_zero_scale_c(dtype):
    out_dt = OUT_DTYPE[dtype]
    C0 = (torch.rand(70, 48, generator=torch.Generator().manual_seed(3)) * 2 - 1).to(out_dt)
    A = torch.empty(70, 8, dtype=G_in(dtype), device="cuda")
    B = torch.empty(8, 48, dtype=G_in(dtype), device="cuda")
    for K in (0, 8):
        C = C0.cuda()
        Ak = A[:, :K] if K else torch.empty(70, 0, dtype=A.dtype, device="cuda")
        Bk = B[:K] if K else torch.empty(0, 48, dtype=B.dtype, device="cuda")
        if K:
            Ak.fill_(float("inf"))          # alpha == 0 must not read A or B
        G.gemm(Ak, Bk, C, 0.0 if K else 1.0, -0.5, stages=2, checked=True)
        expect = (-0.5 * C0.double()).to(out_dt).double()
        assert torch.equal(C.double().cpu(), expect)


def G_in(dtype):
    from stage_software_pipelining_gb300.workloads import IN_DTYPE
    return IN_DTYPE[dtype]


def test_automatic_tile_choice_on_gb300():
    """The automatic tile on this GPU: the pair tile once the pair tiles fill
    more than half the SMs (or K is long), its 512-wide form when K >= 8192
    and the wide tiles fill a round of pairs, 128 x 256 for one partial round
    at K <= 4096, 128 x 128 when the pair tiles would busy at most a quarter."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sms >= 128
    dt = GEMM_BF16_F32
    assert G.resolve_tile(8192, 8192, 8192, dt) == G.TILE_256x512_2SM
    assert G.resolve_tile(4096, 4096, 8192, dt) == G.TILE_256x512_2SM   # 128 wide tiles
    assert G.resolve_tile(8192, 8192, 4096, dt) == G.TILE_256x256_2SM
    assert G.resolve_tile(2048, 2048, 2048, dt) == G.TILE_128x256     # 64 pair tiles
    assert G.resolve_tile(2048, 2048, 8192, dt) == G.TILE_256x256_2SM
    assert G.resolve_tile(1024, 1024, 4096, dt) == G.TILE_128x128     # 16 pair tiles
    assert G.resolve_tile(8191, 28672, 4096, GEMM_BF16_BF16) == G.TILE_256x256_2SM
    # rings of 5 or 6 stages take the tile of the same rows per SM that holds them
    assert G.resolve_tile(8192, 8192, 8192, dt, stages=6) == G.TILE_256x256_2SM
    assert G.resolve_tile(2048, 2048, 2048, dt, stages=5) == G.TILE_256x256_2SM
    assert G.resolve_tile(1024, 1024, 4096, dt, stages=6) == G.TILE_128x128
    assert G.resolve_tile(100, 2048, 512, dt, stages=6) == G.TILE_128x128


@pytest.mark.parametrize("dtype", [GEMM_BF16_F32, GEMM_BF16_BF16])
def test_automatic_six_stage_ring_is_bitwise_the_pair_tile(dtype):
    """Asking for 6 stages without a tile, where a 4-stage ring would take the
    256 x 512 tile (which holds 4), runs the 256 x 256 pair tile: the same
    bits as either tile at any depth, and within the oracle's tolerance."""
    M, N, K = 2048, 4864, 8192                     # 80 wide tiles on 76 pairs
    assert G.resolve_tile(M, N, K, dtype, stages=4) == G.TILE_256x512_2SM
    assert G.resolve_tile(M, N, K, dtype, stages=6) == G.TILE_256x256_2SM
    w = workload(dtype, M, N, K, beta=0.0)
    inp = make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    out_dt = OUT_DTYPE[dtype]
    outs = {}
    for key, stages, tile in (("auto6", 6, G.TILE_AUTO), ("pair2", 2, G.TILE_256x256_2SM),
                              ("wide4", 4, G.TILE_256x512_2SM)):
        outs[key] = torch.full((M, N), float("nan"), dtype=out_dt, device="cuda")
        G.gemm(A, B, outs[key], 1.0, 0.0, stages=stages, tile=tile, checked=True)
    assert torch.equal(outs["auto6"], outs["pair2"])
    assert torch.equal(outs["auto6"], outs["wide4"])
    rows, cols = sample_indices(M, N, 600, 11)
    got = outs["auto6"][torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
    ref, absb = oracle.gemm_entries(inp.A, inp.B, None, 1.0, 0.0, rows=rows, cols=cols)
    check_against_oracle(got.double().cpu().numpy(), ref, absb, dtype, what="auto 6 stages")


def test_empty_m_or_n_is_a_noop():
    C = torch.full((0, 16), 1.0, device="cuda")
    G.gemm(torch.zeros(0, 8, dtype=torch.bfloat16, device="cuda"),
           torch.zeros(8, 16, dtype=torch.bfloat16, device="cuda"), C, checked=True)


# --------------------------------------------------------------------------- fault path
@pytest.mark.parametrize("tile", [G.TILE_128x128, G.TILE_128x256, G.TILE_256x256_2SM,
                                  G.TILE_256x512_2SM])
def test_withheld_arrive_times_out_and_context_survives(tile):
    """Block 0's producer skips one stage: the MMA wait must run out, the
    kernel must return GEMM_ERR_TIMEOUT (no hang, no trap), and the next
    GEMM on the same context must be correct."""
    inp = make_inputs(workload(GEMM_BF16_F32, 256, 512, 512, beta=0.0))
    A = to_device_padded(inp.A)
    B = to_device_padded(inp.B)
    C = torch.zeros(256, 512, device="cuda")
    try:
        G.debug_set(50_000_000, 3)      # 50 ms per wait; withhold K tile 3
        with pytest.raises(G.GemmError) as e:
            G.gemm(A, B, C, stages=2, tile=tile, checked=True)
        assert e.value.status == G.GEMM_ERR_TIMEOUT
    finally:
        G.debug_set(0, -1)
    G.gemm(A, B, C, stages=2, tile=tile, checked=True)
    ref, absb = oracle_full(inp)
    check_against_oracle(C.double().cpu().numpy(), ref, absb, GEMM_BF16_F32,
                         what="after timeout")


# --------------------------------------------------------------------------- host entry
@pytest.mark.parametrize("dtype", [GEMM_F32, GEMM_BF16_F32, GEMM_BF16_BF16])
def test_host_entry_matches_device_entry(dtype):
    w = workload(dtype, 190, 264, 96, beta=0.0, b_col_major=(dtype == GEMM_BF16_BF16))
    inp = make_inputs(w)
    out_dev, _ = run_gpu(inp, 2)
    Ch = torch.zeros(190, 264, dtype=OUT_DTYPE[dtype]).pin_memory()
    G.gemm_host(inp.A.pin_memory(), inp.B, Ch, stages=2)
    assert np.array_equal(Ch.double().numpy(), out_dev)


@pytest.mark.parametrize("dtype", [GEMM_F32, GEMM_BF16_F32, GEMM_BF16_BF16])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_host_entry_in_row_panels_matches_device_entry(dtype, beta):
    """Tall problems go through gemm_host in row panels (copies in, GEMM and
    copies back overlapped on three streams): every panel, including a
    ragged last one, gives the same bits as one device-side call."""
    # 2300 rows: 9 panels of 256, the last of 252 rows, for which the automatic
    # tile on its own would differ from the one chosen for the whole call
    M, N, K = 2300, 2304, 200
    w = workload(dtype, M, N, K, beta=beta, b_col_major=(dtype == GEMM_BF16_BF16))
    inp = make_inputs(w)
    if inp.C0 is None:
        inp = dataclasses.replace(inp, C0=torch.zeros(M, N, dtype=OUT_DTYPE[dtype]))
    out_dev, _ = run_gpu(inp, 2, beta=beta)
    Ch = inp.C0.clone().pin_memory()
    hB = inp.B.t().contiguous().pin_memory().t() if w.b_col_major else inp.B.pin_memory()
    if dtype != GEMM_F32:     # the whole call takes the pair tile, a lone last panel would not
        assert G.plan(M, N, K, dtype, 2, w.b_col_major)["cluster"] == 2
        assert G.plan(252, N, K, dtype, 2, w.b_col_major)["cluster"] == 1
    G.gemm_host(inp.A.pin_memory(), hB, Ch, w.alpha, beta, stages=2)
    assert np.array_equal(Ch.double().numpy(), out_dev)
    ref, absb = oracle_full(inp, beta=beta)
    check_against_oracle(Ch.double().numpy(), ref, absb, dtype, beta=beta, C0=inp.C0,
                         what=f"gemm_host panels dt={dtype} beta={beta}")


@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_host_panels_of_a_wide_tile_call_give_its_bits(beta):
    """A long-K call resolves to the 256 x 512 tile, but its 256-row panels
    are too short for a round of those tiles and run the 256 x 256 pair tile
    (at its own stage limit): the bits must still be the device call's."""
    M, N, K = 4096, 4096, 8192    # 128 wide tiles: a round of pairs
    dtype = GEMM_BF16_F32
    assert G.resolve_tile(M, N, K, dtype) == G.TILE_256x512_2SM
    assert G.resolve_tile(M // 16, N, K, dtype) != G.TILE_256x512_2SM
    w = workload(dtype, M, N, K, beta=beta)
    inp = make_inputs(w)
    if inp.C0 is None:
        inp = dataclasses.replace(inp, C0=torch.zeros(M, N, dtype=OUT_DTYPE[dtype]))
    out_dev, _ = run_gpu(inp, 4, tile=G.TILE_256x512_2SM, beta=beta)
    Ch = inp.C0.clone().pin_memory()
    G.gemm_host(inp.A.pin_memory(), inp.B.pin_memory(), Ch, w.alpha, beta, stages=4,
                tile=G.TILE_256x512_2SM)
    assert np.array_equal(Ch.double().numpy(), out_dev)


# --------------------------------------------------------------------------- full-size workloads
def sample_indices(M, N, count, seed):
    rng = np.random.default_rng(seed)
    edge_r = [r for r in (0, 1, 127, 128, M // 2, M - 2, M - 1) if 0 <= r < M]
    edge_c = [c for c in (0, 1, 15, 16, 255, 256, N // 2, N - 2, N - 1) if 0 <= c < N]
    rows = [r for r in edge_r for _ in edge_c]
    cols = [c for _ in edge_r for c in edge_c]
    rows += list(rng.integers(0, M, count))
    cols += list(rng.integers(0, N, count))
    return np.array(rows), np.array(cols)


@pytest.mark.parametrize("name,stages,tile", [
    ("fp32_2048", 2, 0),
    ("fp16_2048", 3, 0),
    ("bf16_8192_beta1", 4, G.TILE_128x256),
    ("bf16_8192_beta1", 4, G.TILE_256x512_2SM),     # the configuration bench.py times
    ("bf16_8192_beta1", 6, G.TILE_256x256_2SM),
    ("bf16_8192_beta1", 6, G.TILE_128x128),
    ("bf16_8192_beta1", 5, 0),                      # automatic tile for a 5-stage ring
    ("bf16_ragged_colB", 4, G.TILE_128x256),
    ("bf16_ragged_colB", 6, G.TILE_256x256_2SM),     # the configuration bench.py times
    ("bf16_ragged_colB", 1, G.TILE_256x256_2SM),
    ("bf16_ragged_colB", 4, G.TILE_256x512_2SM),
])
def test_full_size_workload_sampled(name, stages, tile):
    w = BY_NAME[name]
    inp = make_inputs(w)
    A = inp.A.cuda()
    B = inp.B.t().contiguous().t().cuda() if w.b_col_major else inp.B.cuda()
    assert (B.stride(0) == 1) == w.b_col_major
    C = inp.C0.cuda() if inp.C0 is not None else torch.full((w.M, w.N), float("nan"),
                                                            dtype=OUT_DTYPE[w.dtype], device="cuda")
    G.gemm(A, B, C, w.alpha, w.beta, stages=stages, tile=tile, checked=True)
    rows, cols = sample_indices(w.M, w.N, 3000, 7)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    ref, absb = oracle.gemm_entries(inp.A, inp.B, inp.C0, w.alpha, w.beta, rows=rows, cols=cols)
    c0s = inp.C0[torch.from_numpy(rows), torch.from_numpy(cols)] if inp.C0 is not None else None
    check_against_oracle(got, ref, absb, w.dtype, beta=w.beta, C0=c0s, what=name)
    if w.dtype == GEMM_BF16_BF16:
        # Frobenius criterion on the fp32-output launch of the same kernel
        C32 = torch.empty(w.M, w.N, device="cuda")
        G.gemm(A, B, C32, w.alpha, 0.0, stages=stages, tile=tile, checked=True)
        got32 = C32[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()]
        check_against_oracle(got32.double().cpu().numpy(), ref, absb, GEMM_BF16_F32,
                             what=name + " fp32 twin")


def test_full_size_stage_sweep_is_bitwise_invariant():
    """At the 8192^3 bf16 size, every stage count of each tile gives identical
    bits (the sweep the benchmark times)."""
    w = BY_NAME["bf16_8192_beta1"]
    inp = make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    C0 = inp.C0.cuda()
    for tile in TILES:
        base = None
        for s in TILE_STAGES[tile]:
            C = C0.clone()
            G.gemm(A, B, C, w.alpha, w.beta, stages=s, tile=tile, checked=True)
            if base is None:
                base = C
            else:
                assert torch.equal(C, base), f"tile={tile} stages={s}"


@pytest.mark.parametrize("dtype", TC_DTYPES)
@pytest.mark.parametrize("b_col_major", [False, True])
@pytest.mark.parametrize("beta", [0.0, 1.0, -0.75])
def test_wide_tile_is_bitwise_the_pair_tile(dtype, b_col_major, beta):
    """The 256 x 512 tile issues each output's K = 16 steps in the same order
    as the 256 x 256 pair tile (two N = 256 MMAs per step instead of one), so
    C must come out bit for bit the same, on a ragged shape that leaves
    partial wide tiles in both M and N, with C read back (beta != 0, 1),
    added at L2 (beta = 1, fp32 C) or not read (beta = 0)."""
    w = workload(dtype, 700, 1100, 900, alpha=1.25, beta=beta, b_col_major=b_col_major)
    inp = make_inputs(w)
    pair, _ = run_gpu(inp, 3, tile=G.TILE_256x256_2SM)
    wide, _ = run_gpu(inp, 4, tile=G.TILE_256x512_2SM)
    assert np.array_equal(pair, wide)
    ref, absb = oracle_full(inp)
    check_against_oracle(wide, ref, absb, dtype, beta=beta, C0=inp.C0, what="wide tile")


@pytest.mark.parametrize("tile", [G.TILE_256x256_2SM, G.TILE_256x512_2SM])
def test_back_to_back_launches_are_deterministic(tile):
    """200 launches in a row on one stream (consecutive grids overlap through
    programmatic dependent launch; the 256 x 512 tile also hands its
    accumulator over in halves) leave exactly the bits of one checked call."""
    w = workload(GEMM_BF16_BF16, 2048, 4096, 8192, beta=0.0, b_col_major=False)
    inp = make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    one = torch.empty(w.M, w.N, dtype=torch.bfloat16, device="cuda")
    G.gemm(A, B, one, 1.0, 0.0, stages=G.TILE_MAX_STAGES[tile], tile=tile, checked=True)
    many = torch.empty_like(one)
    for _ in range(200):
        G.gemm(A, B, many, 1.0, 0.0, stages=G.TILE_MAX_STAGES[tile], tile=tile)
    G.gemm(A, B, many, 1.0, 0.0, stages=G.TILE_MAX_STAGES[tile], tile=tile, checked=True)
    assert torch.equal(one, many)


@pytest.mark.parametrize("M,N,K", [(1_048_581, 136, 40),    # 4097 pair-tile rows, ragged
                                   (130, 200, 131_080)])    # 2049 stages of K = 64
def test_extreme_dimensions_sampled(M, N, K):
    """Very tall and very deep problems: tile indices, TMA row coordinates,
    64-bit C offsets and long accumulation chains, checked on sampled
    entries (the oracle computes each one as a K-term dot product)."""
    w = workload(GEMM_BF16_F32, M, N, K, beta=1.0)
    inp = make_inputs(w)
    A, B, C = inp.A.cuda(), inp.B.cuda(), inp.C0.cuda()
    G.gemm(A, B, C, w.alpha, w.beta, checked=True)
    rows, cols = sample_indices(M, N, 1500, seed=11)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    ref, absb = oracle.gemm_entries(inp.A, inp.B, inp.C0, w.alpha, w.beta, rows=rows, cols=cols)
    c0s = inp.C0[torch.from_numpy(rows), torch.from_numpy(cols)]
    # The elementwise bound holds as stated.  The relative Frobenius bound
    # (1e-4) is stated for K up to 8192; rounding in an fp32 accumulation
    # grows like sqrt(K), so it is scaled by sqrt(K / 8192) beyond that.
    check_against_oracle(got, ref, absb, GEMM_BF16_F32, beta=w.beta, C0=c0s,
                         what=f"extreme {M}x{N}x{K}", frob=False)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-4 * max(1.0, np.sqrt(K / 8192)), f"relative Frobenius error {rel:.3e}"


def test_calls_replay_from_a_cuda_graph():
    """gemm enqueues plain kernel launches (no allocation, no host sync on the
    default schedule), so a sequence of calls can be captured into a CUDA
    graph and replayed: three captured C += A*B, replayed twice, give
    C0 + 6*A*B."""
    w = workload(GEMM_BF16_F32, 700, 520, 264, beta=1.0)
    inp = make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    C = inp.C0.cuda()
    G.gemm(A, B, C.clone(), 1.0, 1.0)            # first call outside the capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            G.gemm(A, B, C, 1.0, 1.0, stream=s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    ref, absb = oracle.gemm(inp.A, inp.B, inp.C0, 6.0, 1.0)
    check_against_oracle(C.double().cpu().numpy(), ref, 6.0 * absb, GEMM_BF16_F32, beta=1.0,
                         C0=inp.C0, what="graph replay")


# --------------------------------------------------------------------------- stream-K tail
@pytest.fixture
def stream_k():
    G.schedule_set(G.SCHEDULE_STREAM_K)
    yield
    G.schedule_set(G.SCHEDULE_AUTO)


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("dtype", [GEMM_BF16_F32, GEMM_BF16_BF16, GEMM_F16_F32])
@pytest.mark.parametrize("shape", [(768, 1280, 1024), (300, 520, 2000), (1100, 900, 4096)])
def test_stream_k_matches_oracle(stream_k, tile, dtype, shape):
    """Fewer tiles than persistent units: every tile is cut along K over
    several units (up to ~5 contributors per tile) and reduced by the unit
    that holds k = 0."""
    M, N, K = shape
    inp = make_inputs(workload(dtype, M, N, K, beta=0.0))
    out, _ = run_gpu(inp, 3, tile=tile)
    ref, absb = oracle_full(inp)
    check_against_oracle(out, ref, absb, dtype, what=f"stream-K {shape} tile={tile} dt={dtype}")


@pytest.mark.parametrize("tile", TILES)
def test_stream_k_stage_invariance_and_beta(stream_k, tile):
    w = workload(GEMM_BF16_F32, 700, 1000, 1500, beta=1.0)
    inp = make_inputs(w)
    outs = {s: run_gpu(inp, s, tile=tile)[0] for s in TILE_STAGES[tile]}
    base = outs[TILE_STAGES[tile][0]]
    for s, o in outs.items():
        assert np.array_equal(o, base), f"stream-K stages={s} differs (tile={tile})"
    ref, absb = oracle_full(inp)
    check_against_oracle(base, ref, absb, GEMM_BF16_F32, beta=1.0, C0=inp.C0,
                         what=f"stream-K beta=1 tile={tile}")


def test_stream_k_workspace_reused_across_tiles(stream_k):
    """One stream, one cached workspace, calls with tiles whose partial slots
    differ in size, largest first: each call's flags must start cleared
    wherever an earlier call left its partials."""
    inp = make_inputs(workload(GEMM_BF16_F32, 768, 1280, 1024, beta=0.0))
    ref, absb = oracle_full(inp)
    for tile in (G.TILE_256x512_2SM, G.TILE_256x256_2SM, G.TILE_128x128, G.TILE_128x256,
                 G.TILE_128x128, G.TILE_256x512_2SM):
        out, _ = run_gpu(inp, 2, tile=tile)
        check_against_oracle(out, ref, absb, GEMM_BF16_F32, what=f"stream-K reuse tile={tile}")


def test_stream_k_schedules_agree_within_tolerance():
    inp = make_inputs(workload(GEMM_BF16_F32, 1024, 1536, 2048, beta=0.0))
    ref, absb = oracle_full(inp)
    outs = {}
    try:
        for sched in (G.SCHEDULE_FULL_TILES, G.SCHEDULE_STREAM_K, G.SCHEDULE_AUTO):
            G.schedule_set(sched)
            outs[sched], _ = run_gpu(inp, 3, tile=G.TILE_256x256_2SM)
            check_against_oracle(outs[sched], ref, absb, GEMM_BF16_F32, what=f"schedule {sched}")
    finally:
        G.schedule_set(G.SCHEDULE_AUTO)


@pytest.mark.parametrize("tile", [G.TILE_128x256, G.TILE_256x256_2SM, G.TILE_256x512_2SM])
def test_stream_k_timeout_leaves_context_usable(stream_k, tile):
    inp = make_inputs(workload(GEMM_BF16_F32, 512, 768, 1024, beta=0.0))
    A = to_device_padded(inp.A)
    B = to_device_padded(inp.B)
    C = torch.zeros(512, 768, device="cuda")
    try:
        # under stream-K block 0 may own a single K iteration: withhold the first
        G.debug_set(50_000_000, 0)
        with pytest.raises(G.GemmError) as e:
            G.gemm(A, B, C, stages=2, tile=tile, checked=True)
        assert e.value.status == G.GEMM_ERR_TIMEOUT
    finally:
        G.debug_set(0, -1)
    G.gemm(A, B, C, stages=2, tile=tile, checked=True)
    ref, absb = oracle_full(inp)
    check_against_oracle(C.double().cpu().numpy(), ref, absb, GEMM_BF16_F32,
                         what="stream-K after timeout")


# --------------------------------------------------------------------------- streams
def test_launch_goes_on_the_callers_stream():
    """gemm enqueues on the stream it is given: work queued before it on that
    stream is finished first, and an event recorded after it completes after."""
    w = workload(GEMM_BF16_F32, 512, 512, 512, beta=1.0)
    inp = make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    s = torch.cuda.Stream()
    C = torch.empty(512, 512, device="cuda")
    with torch.cuda.stream(s):
        C.copy_(inp.C0.cuda(non_blocking=False))   # queued on s before the GEMM
        G.gemm(A, B, C, 1.0, 1.0, stages=3, tile=G.TILE_256x256_2SM, stream=s)
        done = torch.cuda.Event()
        done.record(s)
    done.synchronize()
    ref, absb = oracle_full(inp)
    check_against_oracle(C.double().cpu().numpy(), ref, absb, GEMM_BF16_F32, beta=1.0,
                         C0=inp.C0, what="non-default stream")


@pytest.mark.parametrize("schedule", [G.SCHEDULE_AUTO, G.SCHEDULE_STREAM_K])
def test_concurrent_streams(schedule):
    """Two GEMMs queued on two streams at once (their kernels may overlap on
    the GPU) write their own C correctly; under stream-K each stream has its
    own workspace."""
    w1 = workload(GEMM_BF16_F32, 1100, 904, 2048, beta=1.0)
    w2 = workload(GEMM_BF16_BF16, 700, 1000, 1504, beta=0.0)
    in1, in2 = make_inputs(w1), make_inputs(w2)
    A1, B1, C1 = in1.A.cuda(), in1.B.cuda(), in1.C0.cuda()
    A2 = in2.A.cuda()
    B2 = in2.B.t().contiguous().t().cuda() if w2.b_col_major else in2.B.cuda()
    C2 = torch.zeros(700, 1000, dtype=torch.bfloat16, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    try:
        G.schedule_set(schedule)
        for _ in range(3):                      # C1 accumulates three products
            G.gemm(A1, B1, C1, 1.0, 1.0, stream=s1)
            G.gemm(A2, B2, C2, 1.0, 0.0, stream=s2)
        torch.cuda.synchronize()
    finally:
        G.schedule_set(G.SCHEDULE_AUTO)
    ref1, absb1 = oracle.gemm(in1.A, in1.B, in1.C0, 3.0, 1.0)
    check_against_oracle(C1.double().cpu().numpy(), ref1, 3.0 * absb1, GEMM_BF16_F32, beta=1.0,
                         C0=in1.C0, what=f"stream 1, schedule {schedule}")
    ref2, absb2 = oracle.gemm(in2.A, in2.B, None, 1.0, 0.0)
    check_against_oracle(C2.double().cpu().numpy(), ref2, absb2, GEMM_BF16_BF16,
                         what=f"stream 2, schedule {schedule}")


def test_release_then_reuse():
    G.load_library().gemm_host_release()
    inp = make_inputs(workload(GEMM_BF16_F32, 256, 256, 256, beta=0.0))
    out, _ = run_gpu(inp, 2)
    ref, absb = oracle_full(inp)
    check_against_oracle(out, ref, absb, GEMM_BF16_F32, what="after release")
