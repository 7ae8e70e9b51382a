"""Pins for the CPU oracle (no GPU).

The oracle is the plain fp64 definition C = alpha*A*B + beta*C0 (the problem
"CUTLASS-CuTe 初步(6)", section 2 "Thread Block Tile", states as C += A*B over
the K tiles).  These tests tie it to things other than itself: hand-worked
fixtures under tests/golden/, identities, a closed form, exact rational
arithmetic on tiny shapes, library routines (numpy's float16 and fp64 matmul,
torch's bfloat16), and a mutation check showing that a planted mistake in a
copy of the oracle (a sign, a dropped term, a transposed operand, a wrong
decode) fails at least one of these pins.
"""
import os
import re
import shutil
import subprocess
import sys
from fractions import Fraction

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import oracle  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


# ----------------------------------------------------------------------------- helpers
def parse_fixture(path):
    """Parse a golden fixture: header keys, then named matrices."""
    meta, mats = {}, {}
    lines = [ln.strip() for ln in open(path, encoding="utf-8")]
    lines = [ln for ln in lines if ln and not ln.startswith("#")]
    i = 0
    while i < len(lines):
        parts = lines[i].split()
        if len(parts) == 3 and parts[1].isdigit() and parts[2].isdigit():
            name, r, c = parts[0], int(parts[1]), int(parts[2])
            rows = [[float(v) for v in lines[i + 1 + t].split()] for t in range(r)]
            assert all(len(row) == c for row in rows), (path, name)
            mats[name] = np.array(rows, dtype=np.float64)
            i += 1 + r
        else:
            meta[parts[0]] = parts[1]
            i += 1
    return meta, mats


def as_storage(x, dt, col_major=False):
    """Host tensor of dtype dt holding x exactly (asserts exactness)."""
    t = torch.tensor(np.asarray(x, dtype=np.float64)).to(TORCH_DT[dt])
    assert torch.equal(t.double(), torch.tensor(np.asarray(x, dtype=np.float64))), \
        "fixture value not exact in storage type"
    if col_major:
        t = t.t().contiguous().t()       # same logical matrix, column-major storage
    return t


def rand_int(gen, shape, lo=-3, hi=3):
    return torch.randint(lo, hi + 1, shape, generator=gen).to(torch.float32)


# ----------------------------------------------------------------------------- fixtures
FIXTURES = sorted(f for f in os.listdir(GOLDEN) if f.startswith("gemm_") and f.endswith(".txt"))


def check_fixture(fname):
    meta, m = parse_fixture(os.path.join(GOLDEN, fname))
    dt = meta["dtype"]
    A = as_storage(m["A"], dt)
    B = as_storage(m["B"], dt, col_major=meta["b_layout"] == "col")
    alpha, beta = float(meta["alpha"]), float(meta["beta"])
    C0 = as_storage(m["C0"], "f32") if "C0" in m else None
    C, Abs = oracle.gemm(A, B, C0, alpha, beta)
    assert np.array_equal(C, m["C"]), (fname, C, m["C"])
    if "Abs" in m:
        assert np.array_equal(Abs, m["Abs"]), (fname, Abs, m["Abs"])


def test_fixture_files_present():
    assert len(FIXTURES) >= 4


@pytest.mark.parametrize("fname", FIXTURES)
def test_golden_fixture(fname):
    check_fixture(fname)


# ----------------------------------------------------------------------------- decoders
def check_decode_f16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)          # numpy's IEEE binary16
    got = np.array([oracle.decode_f16(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def check_decode_bf16_all_patterns():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double().numpy()          # torch's bfloat16
    got = np.array([oracle.decode_bf16(int(b) & 0xFFFF) for b in bits.tolist()])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_decode_f16_all_patterns():
    check_decode_f16_all_patterns()


def test_decode_bf16_all_patterns():
    check_decode_bf16_all_patterns()


def test_decode_f32_patterns():
    rng = np.random.default_rng(7)
    special = np.array([0, 0x80000000, 1, 0x007FFFFF, 0x00800000, 0x3F800000, 0xBF800000,
                        0x7F7FFFFF, 0x7F800000, 0xFF800000, 0x7FC00000, 0x34000000],
                       dtype=np.uint32)
    bits = np.concatenate([special, rng.integers(0, 2**32, 20000, dtype=np.uint64)
                           .astype(np.uint32)])
    ref = bits.view(np.float32).astype(np.float64)            # numpy's IEEE binary32
    got = np.array([oracle.decode_f32(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ----------------------------------------------------------------------------- identities
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("col", [False, True])
def test_identity_right_and_left(dt, col):
    check_identities(dt, col)


def check_identities(dt, col):
    gen = torch.Generator().manual_seed(11)
    A = (torch.randn(13, 9, generator=gen)).to(TORCH_DT[dt])
    I9 = torch.eye(9).to(TORCH_DT[dt])
    I13 = torch.eye(13).to(TORCH_DT[dt])
    if col:
        I9 = I9.t().contiguous().t()
    C, _ = oracle.gemm(A, I9)                       # A * I = A
    assert np.array_equal(C, A.double().numpy())
    B = torch.randn(13, 9, generator=gen).to(TORCH_DT[dt])
    if col:
        B = B.t().contiguous().t()
    C, _ = oracle.gemm(I13, B)                      # I * B = B
    assert np.array_equal(C, B.double().numpy())


def check_alpha_zero_and_zero_matrix():
    gen = torch.Generator().manual_seed(12)
    A = torch.randn(7, 5, generator=gen)
    B = torch.randn(5, 6, generator=gen)
    C0 = torch.randn(7, 6, generator=gen)
    C, _ = oracle.gemm(A, B, C0, alpha=0.0, beta=-0.75)
    assert np.array_equal(C, -0.75 * C0.double().numpy())
    C, _ = oracle.gemm(torch.zeros(7, 5), B, C0, alpha=1.5, beta=2.0)
    assert np.array_equal(C, 2.0 * C0.double().numpy())


def test_alpha_zero_and_zero_matrix_give_beta_c():
    check_alpha_zero_and_zero_matrix()


def check_beta_zero_ignores_c0():
    gen = torch.Generator().manual_seed(13)
    A = torch.randn(4, 3, generator=gen)
    B = torch.randn(3, 5, generator=gen)
    C0 = torch.full((4, 5), float("nan"))
    C, _ = oracle.gemm(A, B, C0, alpha=1.0, beta=0.0)
    assert np.isfinite(C).all()
    ref, _ = oracle.gemm(A, B)
    assert np.array_equal(C, ref)


def test_beta_zero_does_not_read_c0():
    check_beta_zero_ignores_c0()


def test_power_of_two_scaling_is_exact():
    gen = torch.Generator().manual_seed(14)
    A = torch.randn(6, 8, generator=gen)
    B = torch.randn(8, 4, generator=gen)
    C1, _ = oracle.gemm(A, B, alpha=1.0)
    C4, _ = oracle.gemm(A, B, alpha=4.0)
    assert np.array_equal(C4, 4.0 * C1)
    C2, _ = oracle.gemm(A * 2, B)
    assert np.array_equal(C2, 2.0 * C1)


def check_associativity_integer():
    """(A*B)*x == A*(B*x) exactly, for small integers (all sums exact)."""
    gen = torch.Generator().manual_seed(15)
    A = rand_int(gen, (6, 5))
    B = rand_int(gen, (5, 7))
    x = rand_int(gen, (7, 1))
    AB, _ = oracle.gemm(A, B)
    left, _ = oracle.gemm(torch.tensor(AB, dtype=torch.float32), x)
    Bx, _ = oracle.gemm(B, x)
    right, _ = oracle.gemm(A, torch.tensor(Bx, dtype=torch.float32))
    assert np.array_equal(left, right)
    # and both equal the integer product computed with Python ints
    Ai = [[int(v) for v in r] for r in A.tolist()]
    Bi = [[int(v) for v in r] for r in B.tolist()]
    xi = [int(v[0]) for v in x.tolist()]
    ABi = [[sum(Ai[i][k] * Bi[k][j] for k in range(5)) for j in range(7)] for i in range(6)]
    exact = [sum(ABi[i][j] * xi[j] for j in range(7)) for i in range(6)]
    assert left[:, 0].tolist() == exact


def test_associativity_integer():
    check_associativity_integer()


def test_associativity_random_real():
    """(A*B)*x vs A*(B*x) with real inputs: agree to fp64 rounding.

    The oracle reads only fp32/fp16/bf16 storage, so the inner product is fed
    back through numpy fp64 for the second multiplication on both sides."""
    gen = torch.Generator().manual_seed(16)
    A = torch.randn(20, 30, generator=gen)
    B = torch.randn(30, 25, generator=gen)
    x = torch.randn(25, generator=gen).double().numpy()
    AB, _ = oracle.gemm(A, B)
    left = AB @ x
    Bn = B.double().numpy()
    right = A.double().numpy() @ (Bn @ x)
    scale = np.abs(A.double().numpy()) @ (np.abs(Bn) @ np.abs(x))
    assert np.all(np.abs(left - right) <= 1e-12 * scale)


# ----------------------------------------------------------------------------- closed forms
def check_rank1_closed_form():
    """A = u*1^T, B = 1*v^T  ->  C_ij = K*u_i*v_j exactly."""
    gen = torch.Generator().manual_seed(17)
    M, N, K = 9, 11, 37
    u = rand_int(gen, (M, 1), -5, 5)
    v = rand_int(gen, (1, N), -5, 5)
    A = u.expand(M, K).contiguous().to(torch.bfloat16)
    B = v.expand(K, N).contiguous().to(torch.bfloat16)
    C, Abs = oracle.gemm(A, B)
    expect = K * u.double().numpy() @ v.double().numpy()
    assert np.array_equal(C, expect)
    assert np.array_equal(Abs, np.abs(expect))


def test_rank1_closed_form():
    check_rank1_closed_form()


def test_all_ones_gives_k():
    for K in (1, 5, 64, 257):
        C, Abs = oracle.gemm(torch.ones(3, K, dtype=torch.float16),
                             torch.ones(K, 4, dtype=torch.float16))
        assert np.all(C == K) and np.all(Abs == K)
        C, Abs = oracle.gemm(torch.ones(3, K), -torch.ones(K, 4))
        assert np.all(C == -K) and np.all(Abs == K)


# ----------------------------------------------------------------------------- brute force
def frac_gemm(A, B, C0, alpha, beta):
    M, K = len(A), len(A[0]) if A else 0
    N = len(B[0]) if B else 0
    out = []
    for i in range(M):
        row = []
        for j in range(N):
            s = sum((Fraction(A[i][k]) * Fraction(B[k][j]) for k in range(K)), Fraction(0))
            v = Fraction(alpha) * s
            if beta != 0:
                v += Fraction(beta) * Fraction(C0[i][j])
            row.append(v)
        out.append(row)
    return out


def check_bruteforce_fraction(seed_count=60):
    rng = np.random.default_rng(18)
    for trial in range(seed_count):
        M, N, K = (int(v) for v in rng.integers(1, 5, 3))
        dt = ["f32", "f16", "bf16"][trial % 3]
        col = bool(trial % 2)
        alpha = float(rng.choice([1.0, -0.5, 2.0, 0.375]))
        beta = float(rng.choice([0.0, 1.0, -1.25]))
        gen = torch.Generator().manual_seed(100 + trial)
        A = torch.randn(M, K, generator=gen).to(TORCH_DT[dt])
        Bl = torch.randn(K, N, generator=gen).to(TORCH_DT[dt])
        B = Bl.t().contiguous().t() if col else Bl
        C0 = torch.randn(M, N, generator=gen)
        C, Abs = oracle.gemm(A, B, C0, alpha, beta)
        Ad = A.double().tolist()
        Bd = Bl.double().tolist()
        exact = frac_gemm(Ad, Bd, C0.double().tolist(), alpha, beta)
        for i in range(M):
            for j in range(N):
                e = exact[i][j]
                bound = (abs(alpha) * Abs[i, j] + abs(beta) * abs(float(C0[i, j]))) \
                    * (K + 2) * 2.0 ** -52
                assert abs(Fraction(C[i, j]) - e) <= Fraction(bound), (trial, i, j)
                abs_exact = sum(abs(Fraction(Ad[i][k]) * Fraction(Bd[k][j])) for k in range(K))
                assert abs(Fraction(Abs[i, j]) - abs_exact) <= Fraction(K * 2.0 ** -52 *
                                                                        Abs[i, j])


def test_bruteforce_fraction_tiny_shapes():
    check_bruteforce_fraction()


# ----------------------------------------------------------------------------- library routine
@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("col", [False, True])
def test_matches_numpy_fp64_matmul(dt, col):
    check_numpy(dt, col)


def check_numpy(dt="f32", col=False):
    gen = torch.Generator().manual_seed(19)
    M, N, K = 37, 53, 61
    A = torch.randn(M, K, generator=gen).to(TORCH_DT[dt])
    Bl = torch.randn(K, N, generator=gen).to(TORCH_DT[dt])
    B = Bl.t().contiguous().t() if col else Bl
    C0 = torch.randn(M, N, generator=gen)
    C, Abs = oracle.gemm(A, B, C0, 1.25, -0.5)
    An, Bn = A.double().numpy(), Bl.double().numpy()
    ref = 1.25 * (An @ Bn) - 0.5 * C0.double().numpy()
    absref = np.abs(An) @ np.abs(Bn)
    assert np.all(np.abs(C - ref) <= 1e-13 * (absref + np.abs(C0.double().numpy())))
    assert np.allclose(Abs, absref, rtol=1e-14, atol=0)


def test_padded_leading_dimensions():
    gen = torch.Generator().manual_seed(20)
    A_big = torch.randn(10, 16, generator=gen).to(torch.bfloat16)
    B_big = torch.randn(7, 24, generator=gen).to(torch.bfloat16)
    C0_big = torch.randn(10, 32, generator=gen)
    A, B, C0 = A_big[:, :7], B_big[:, :11], C0_big[:, :11]
    assert A.stride() == (16, 1) and B.stride() == (24, 1)
    C, _ = oracle.gemm(A, B, C0, 1.0, 1.0)
    Cc, _ = oracle.gemm(A.contiguous(), B.contiguous(), C0.contiguous(), 1.0, 1.0)
    assert np.array_equal(C, Cc)
    # column-major B with padding: (K x N) view of an N x ldb buffer
    Bcm_big = torch.randn(11, 12, generator=gen).to(torch.bfloat16)
    Bcm = Bcm_big[:, :7].t()
    assert Bcm.stride() == (1, 12)
    C, _ = oracle.gemm(A, Bcm)
    Cc, _ = oracle.gemm(A, Bcm.contiguous())
    assert np.array_equal(C, Cc)


def test_rows_and_entries_agree_with_full():
    gen = torch.Generator().manual_seed(21)
    A = torch.randn(23, 17, generator=gen).to(torch.float16)
    B = torch.randn(17, 29, generator=gen).to(torch.float16).t().contiguous().t()
    C0 = torch.randn(23, 29, generator=gen)
    C, Abs = oracle.gemm(A, B, C0, 0.5, 2.0)
    Cs, Abss = oracle.gemm(A, B, C0, 0.5, 2.0, rows=(5, 12))
    assert np.array_equal(Cs, C[5:12]) and np.array_equal(Abss, Abs[5:12])
    r = np.array([0, 22, 7, 13])
    c = np.array([28, 0, 3, 13])
    v, a = oracle.gemm_entries(A, B, C0, 0.5, 2.0, rows=r, cols=c)
    assert np.array_equal(v, C[r, c]) and np.array_equal(a, Abs[r, c])


def test_threads_do_not_change_bits():
    gen = torch.Generator().manual_seed(22)
    A = torch.randn(33, 40, generator=gen)
    B = torch.randn(40, 19, generator=gen)
    C1, _ = oracle.gemm(A, B, nthreads=1)
    C4, _ = oracle.gemm(A, B, nthreads=4)
    assert np.array_equal(C1, C4)


def test_degenerate_sizes():
    C, Abs = oracle.gemm(torch.zeros(0, 5), torch.zeros(5, 3))
    assert C.shape == (0, 3)
    C0 = torch.randn(4, 3)
    C, Abs = oracle.gemm(torch.zeros(4, 0), torch.zeros(0, 3), C0, 1.0, 0.5)
    assert np.array_equal(C, 0.5 * C0.double().numpy()) and np.all(Abs == 0)
    C, Abs = oracle.gemm(torch.zeros(4, 0), torch.zeros(0, 3))
    assert np.all(C == 0)


def test_argument_errors():
    lib = oracle._load()
    a = np.zeros(16, dtype=np.float32)
    out = np.zeros(16)
    p = a.ctypes.data
    # negative size, ld too small, bad type code
    assert lib.oracle_gemm_rows(-1, 2, 2, p, 2, 0, p, 2, 0, 0, None, 2, 0, 1.0, 0.0,
                                out.ctypes.data, 2, None, 2, 0, 0, 1) == -1
    assert lib.oracle_gemm_rows(2, 2, 4, p, 3, 0, p, 2, 0, 0, None, 2, 0, 1.0, 0.0,
                                out.ctypes.data, 2, None, 2, 0, 2, 1) == -1
    assert lib.oracle_gemm_rows(2, 2, 2, p, 2, 7, p, 2, 0, 0, None, 2, 0, 1.0, 0.0,
                                out.ctypes.data, 2, None, 2, 0, 2, 1) == -1
    # beta != 0 with no C0
    assert lib.oracle_gemm_rows(2, 2, 2, p, 2, 0, p, 2, 0, 0, None, 2, 0, 1.0, 1.0,
                                out.ctypes.data, 2, None, 2, 0, 2, 1) == -1
    with pytest.raises(ValueError):
        oracle.gemm(torch.zeros(2, 3), torch.zeros(4, 2))


# ----------------------------------------------------------------------------- mutations
# Each pin check below runs against the module-level oracle library.
PIN_CHECKS = [
    lambda: [check_fixture(f) for f in FIXTURES],
    check_decode_f16_all_patterns,
    check_decode_bf16_all_patterns,
    lambda: check_identities("bf16", True),
    lambda: check_identities("f16", False),
    check_alpha_zero_and_zero_matrix,
    check_beta_zero_ignores_c0,
    check_associativity_integer,
    check_rank1_closed_form,
    lambda: check_bruteforce_fraction(12),
    lambda: check_numpy("f32", False),
    lambda: check_numpy("bf16", True),
]

# (description, regex on the oracle source, replacement): plausible mistakes.
MUTATIONS = [
    ("sign of the product", r"acc\[j\] \+= a \* b;", "acc[j] -= a * b;"),
    ("transposed row-major B", r"k \* ldb \+ j", "j * ldb + k"),
    ("transposed column-major B", r"j \* ldb \+ k :", "k * ldb + j :"),
    ("A indexed by column", r"load\(A, a_type, i \* lda \+ k\)",
     "load(A, a_type, k * lda + i)"),
    ("beta term dropped", r"if \(beta != 0\.0\) out \+= beta \*", "if (0) out += beta *"),
    ("alpha dropped", r"double out = alpha \* acc\[j\];", "double out = acc[j];"),
    ("beta read although zero", r"if \(beta != 0\.0\) out \+=", "out +="),
    ("bf16 exponent bias", r"e - 134", "e - 133"),
    ("fp16 subnormal scale", r"ldexp\(\(double\)f, -24\)", "ldexp((double)f, -25)"),
    ("fp16 hidden bit", r"1024 \+ f", "f"),
    ("first k skipped", r"for \(int64_t k = 0; k < K; \+\+k\) \{\n                double a",
     "for (int64_t k = 1; k < K; ++k) {\n                double a"),
]


@pytest.mark.parametrize("desc,pattern,repl", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_reject_planted_mistake(tmp_path, desc, pattern, repl):
    src = open(oracle._SRC, encoding="utf-8").read()
    mutated, n = re.subn(pattern, repl, src, count=1)
    assert n == 1, f"mutation pattern for '{desc}' no longer matches the oracle source"
    path = tmp_path / "mut.c"
    path.write_text(mutated, encoding="utf-8")
    so = str(tmp_path / "libmut.so")
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                    "-o", so, str(path), "-lm"], check=True)
    # A mutant may read out of bounds and crash, so its pins run in a child
    # process; a crash counts as caught.  The child's exit code is the number
    # of pin checks that failed.
    env = dict(os.environ, OMP_NUM_THREADS="2")
    proc = subprocess.run([sys.executable, os.path.abspath(__file__), so], env=env,
                          capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, f"no pin caught the planted mistake: {desc}"


def run_pins_against(so_path):
    """Run every pin check against another oracle build; return failures."""
    failures = 0
    with oracle.using_library(so_path):
        for check in PIN_CHECKS:
            try:
                check()
            except (AssertionError, RuntimeError, ValueError):
                failures += 1
    return failures


def test_unmutated_oracle_passes_all_pin_checks():
    for check in PIN_CHECKS:
        check()


def test_gcc_available():
    assert shutil.which("gcc") is not None


if __name__ == "__main__":
    sys.exit(min(run_pins_against(sys.argv[1]), 100))


# ----------------------------------------------------------------------------- streaming copy
def test_copy_oracle_is_byte_identity():
    """The streaming copy's definition: byte i of the output is byte i of the
    input (checked against numpy's own copy and the input itself)."""
    rng = np.random.default_rng(23)
    for n in (0, 1, 15, 16, 4096 + 7):
        src = rng.integers(0, 256, n, dtype=np.uint8)
        out = oracle.copy_bytes(src)
        assert out.dtype == np.uint8 and out.shape == src.shape
        assert np.array_equal(out, src.copy())
        if n:
            assert out.ctypes.data != src.ctypes.data
