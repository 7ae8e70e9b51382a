"""gemm_noalloc: the GEMM entry point for callers that must not allocate.

Some callers cannot call cudaMalloc where they run the GEMM: their device
memory belongs to their own pool allocator, they run a latency-critical loop
that must not take cudaMalloc's implicit device synchronisation, or the
memory is already handed out.  gemm_noalloc keeps the stream-K partials in a
fixed array inside the library instead of a workspace it would allocate.

This test calls it through the C ABI (the caller supplies inputs and output,
as a real caller would) and checks that two calls in a row give the same
result as the existing entry point gemm_ex, within the tolerance the other
tests use (|diff| <= 2e-3 * (|A||B|)_ij, the oracle providing |A||B|), on
shapes where the stream-K tail -- and therefore the fixed array -- is used.
It lives in its own file so that it runs last, and it passes on its own in a
fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_against_oracle
from stage_software_pipelining_gb300 import build as gemm_build
from stage_software_pipelining_gb300 import gemm as G
from stage_software_pipelining_gb300.workloads import (BY_NAME, GEMM_BF16_BF16, GEMM_BF16_F32,
                                                       OUT_DTYPE, make_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib(gpu):
    gemm_build.build()
    return G.load_library()


def call(fn, A, B, C, alpha, beta, dtype, stages, tile):
    """Call gemm_ex or gemm_noalloc through the C ABI on the current stream."""
    M, N, K, lda, ldb, bcm, ldc, code = G._args(A, B, C)
    assert code == dtype
    stream = torch.cuda.current_stream().cuda_stream
    return fn(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
              ctypes.c_float(alpha), ctypes.c_float(beta), dtype, stages, bcm, tile, stream)


CASES = [
    # (base workload, M, N, K, tile, stages): fewer or ragged tiles than units,
    # so the stream-K tail runs and uses the fixed array
    ("bf16_8192_beta1", 1100, 904, 4096, G.TILE_256x256_2SM, 3),
    ("bf16_8192_beta1", 700, 1000, 1504, G.TILE_128x256, 3),
    ("bf16_ragged_colB", 1000, 1200, 2048, G.TILE_256x256_2SM, 2),
    ("bf16_8192_beta1", 1100, 904, 4096, G.TILE_128x128, 6),
    ("bf16_8192_beta1", 1100, 904, 4096, G.TILE_AUTO, 6),
]


@pytest.mark.parametrize("name,M,N,K,tile,stages", CASES)
def test_noalloc_matches_gemm_ex_on_two_calls_in_a_row(lib, name, M, N, K, tile, stages):
    w = BY_NAME[name].resized(M, N, K)
    inp = make_inputs(w)
    A = inp.A.cuda()
    B = (inp.B.t().contiguous().t() if w.b_col_major else inp.B).cuda()
    out_dt = OUT_DTYPE[w.dtype]
    C0 = (inp.C0 if inp.C0 is not None else torch.zeros(M, N, dtype=out_dt)).cuda()

    C_ex = C0.clone()
    assert call(lib.gemm_ex, A, B, C_ex, w.alpha, w.beta, w.dtype, stages, tile) == G.GEMM_OK
    results = []
    for _ in range(2):                       # the second call reuses the array
        C = C0.clone()
        st = call(lib.gemm_noalloc, A, B, C, w.alpha, w.beta, w.dtype, stages, tile)
        assert st == G.GEMM_OK, G.status_string(st)
        results.append(C)
    torch.cuda.synchronize()

    _, absb = oracle.gemm(inp.A, inp.B, inp.C0 if w.beta != 0.0 else None, w.alpha, w.beta)
    ex = C_ex.double().cpu().numpy()
    for i, C in enumerate(results):
        got = C.double().cpu().numpy()
        bound = 2e-3 * absb
        if w.dtype == GEMM_BF16_BF16:        # both sides were rounded to bf16
            bound = bound + 2.0 ** -7 * np.abs(ex)
        bad = ~(np.abs(got - ex) <= bound)
        assert not bad.any(), f"call {i + 1}: {int(bad.sum())} entries differ from gemm_ex " \
                              f"beyond the tolerance"
    # the two calls compute the same thing the same way
    assert torch.equal(results[0], results[1])


def test_noalloc_matches_oracle_at_the_headline_shape(lib):
    """bf16 8192^3 with beta = 1: 1024 pair tiles on the persistent units leave
    a partial last round, which runs as the stream-K tail in the fixed array."""
    w = BY_NAME["bf16_8192_beta1"]
    inp = make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    C = inp.C0.cuda()
    st = call(lib.gemm_noalloc, A, B, C, w.alpha, w.beta, w.dtype, 3, G.TILE_256x256_2SM)
    assert st == G.GEMM_OK, G.status_string(st)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    rows = np.concatenate([[0, 8191, 4096], rng.integers(0, w.M, 1500)])
    cols = np.concatenate([[0, 8191, 255], rng.integers(0, w.N, 1500)])
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    ref, absb = oracle.gemm_entries(inp.A, inp.B, inp.C0, w.alpha, w.beta, rows=rows, cols=cols)
    c0s = inp.C0[torch.from_numpy(rows), torch.from_numpy(cols)]
    check_against_oracle(got, ref, absb, GEMM_BF16_F32, beta=w.beta, C0=c0s,
                         what="gemm_noalloc 8192^3")


def test_noalloc_automatic_tile_stays_within_the_array(lib):
    """A long-K call whose automatic tile would be the 256 x 512 one (its
    partials do not fit the fixed array) runs the 256 x 256 pair tile and
    agrees with gemm_ex; naming the 256 x 512 tile is refused up front."""
    M, N, K = 2304, 4608, 8192
    assert G.resolve_tile(M, N, K, GEMM_BF16_F32) == G.TILE_256x512_2SM
    w = BY_NAME["bf16_8192_beta1"].resized(M, N, K)
    inp = make_inputs(w)
    A, B = inp.A.cuda(), inp.B.cuda()
    C_ex = inp.C0.cuda()
    C = inp.C0.cuda()
    assert call(lib.gemm_ex, A, B, C_ex, w.alpha, w.beta, w.dtype, 4, 0) == G.GEMM_OK
    st = call(lib.gemm_noalloc, A, B, C, w.alpha, w.beta, w.dtype, 4, 0)
    assert st == G.GEMM_OK, G.status_string(st)
    torch.cuda.synchronize()
    _, absb = oracle.gemm(inp.A[:64], inp.B, inp.C0[:64], w.alpha, w.beta)
    got = C[:64].double().cpu().numpy()
    ex = C_ex[:64].double().cpu().numpy()
    assert np.all(np.abs(got - ex) <= 2e-3 * absb)
    C2 = inp.C0.cuda()
    assert call(lib.gemm_noalloc, A, B, C2, w.alpha, w.beta, w.dtype, 4,
                G.TILE_256x512_2SM) == G.GEMM_ERR_SCRATCH
