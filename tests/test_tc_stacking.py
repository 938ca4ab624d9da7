"""The index algebra of the tensor-core GEMV's K stacking, emulated on the CPU (no GPU, no CUDA path).

A packed block of P physical rows stores its weights atom by atom (64 inputs, P rows of 128 bytes each); a ring
chunk holds floor(256 / P) consecutive atoms. An M = 128, K = 16 MMA whose A operand starts at atom a of a
chunk reads the 128 rows that follow in shared memory: atom a's P rows, then atom a + 1's, and so on (rows past
the chunk are whatever the slot holds). Its B operand, N = 16 s rows starting at atom a of the staged
activations, reads the hi / lo columns of atoms a .. a + s - 1. The tile's lanes q*P .. q*P + P - 1 against
columns 16 q .. 16 q + 15 are then row r's partial sums over atom a + q. This test walks the same chunk /
K-part / group structure as the kernel, applies those MMAs to random data (with garbage past each chunk) and
checks that the diagonal blocks, summed over q, give W @ x exactly as the plain product does (float64).
"""
import numpy as np
import pytest

N_COLS = 16  # 8 activation rows as hi / lo column pairs


def stacking_factor(P, nat, ncols=N_COLS, swiglu=False):
    if swiglu or ncols != 16:
        return 1
    return max(1, min(4, 128 // P, nat))


def emulate_block(W, xhl, rng, KP=16):
    """W: [rows, K] weights of one block (rows <= 128), xhl: [16, K] staged activation columns. Returns the
    [rows, 16] accumulator the epilogue reads (diagonal blocks summed)."""
    rows, K = W.shape
    nat = -(-K // 64)
    P = -(-rows // 8) * 8
    Wp = np.zeros((P, nat * 64))
    Wp[:rows, :K] = W
    Xp = np.zeros((N_COLS, nat * 64))
    Xp[:, :K] = xhl
    st = stacking_factor(P, nat)
    atoms_per_chunk = max(1, 256 // P)
    D = np.full((128, N_COLS * st), np.nan)  # TMEM tile: uninitialised until the first MMA
    first = True
    for a0 in range(0, nat, KP):  # K parts
        a1 = min(nat, a0 + KP)
        for c0 in range(a0, a1, atoms_per_chunk):  # ring chunks
            na = min(atoms_per_chunk, a1 - c0)
            # shared memory as the MMA sees it from the chunk start: the chunk's atoms, then garbage
            slot = rng.standard_normal((na * P + 256, 64))
            for j in range(na):
                slot[j * P:(j + 1) * P] = Wp[:, (c0 + j) * 64:(c0 + j + 1) * 64]

            def mma(a, n_atoms_b):
                nonlocal first, D
                A = slot[a * P:a * P + 128]  # 128 rows from atom a on
                B = np.concatenate([Xp[:, (c0 + a + q) * 64:(c0 + a + q + 1) * 64] for q in range(n_atoms_b)])
                prod = A @ B.T  # [128, 16 * n_atoms_b], all four K steps of the atoms at once
                cols = slice(0, N_COLS * n_atoms_b)
                if first:
                    assert n_atoms_b == st, "the first MMA of a block must cover every column of its tile"
                    D[:, cols] = prod
                    first = False
                else:
                    D[:, cols] += prod

            a = 0
            if st > 1:
                while a + st <= na:
                    mma(a, st)
                    a += st
            while a < na:
                mma(a, 1)
                a += 1
    # epilogue: lane q*P + r, columns 16 q .. + 15, summed over q
    out = np.zeros((rows, N_COLS))
    for q in range(st):
        out += D[q * P:q * P + rows, q * N_COLS:(q + 1) * N_COLS]
    return out


@pytest.mark.parametrize("rows,K", [(32, 17408), (40, 17408), (40, 2048), (48, 5120), (56, 6144), (64, 320),
                                    (24, 64), (8, 200), (128, 1024), (104, 5120)])
def test_stacked_mmas_reproduce_the_product(rows, K):
    rng = np.random.default_rng(rows * 100003 + K)
    W = rng.standard_normal((rows, K))
    xhl = rng.standard_normal((N_COLS, K))
    got = emulate_block(W, xhl, rng)
    want = W @ xhl.T
    assert np.allclose(got, want, rtol=1e-10, atol=1e-8)


def test_stacking_factor_rules():
    # 32-40-row shares of the output / down projections stack 4 / 3 atoms; full blocks and SwiGLU never do
    assert stacking_factor(32, 272) == 4 and stacking_factor(40, 272) == 3 and stacking_factor(64, 80) == 2
    assert stacking_factor(128, 80) == 1 and stacking_factor(72, 80) == 1
    assert stacking_factor(32, 272, swiglu=True) == 1 and stacking_factor(32, 272, ncols=32) == 1
    assert stacking_factor(32, 2) == 2  # never more atoms than K has
    # a chunk always holds at least one full stacked group, so the block's first MMA can start every column
    for P in range(8, 65, 8):
        assert max(1, 256 // P) >= stacking_factor(P, 10 ** 6)
