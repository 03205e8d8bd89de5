"""GPU parity of the paired-CTA GEMM (two CTAs of a cluster on one 256-row tile, the paired
tensor-core MMA) against the oracle, through the C ABI, with the pairing forced on.

Same bounds as the single-CTA kernel ([AE] op table row matmul; ‖g − r‖/‖r‖ ≤ 2e-2 and what
the arithmetic allows: bf16 operands are exact in the fp32 products, so fp32 C ≤ 1e-5 and bf16
C ≤ 4e-3).  Each case also checks, from the GEMM launch record, that the paired kernel ran.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import ops as O
from tests.gpu_util import dev, empty, host, norm_err, sync

pytestmark = pytest.mark.gpu

xt = pytest.importorskip("transformer_fwd_bwd_gb300.xt")


def op(X, t):
    return X.T if t else X


@pytest.fixture
def paired():
    """Forces the paired kernel (and a schedule, when asked) for one test; restores both after."""
    xt.gemm_set_pairing(2)

    def sched(mode):
        xt.gemm_set_schedule(mode)
    yield sched
    xt.gemm_set_schedule(0)
    xt.gemm_set_pairing(0)


def records(fn):
    """(tile-width code, schedule code) of each GEMM launch fn made; a paired launch records
    1000 + BN as its tile width."""
    xt.profile_gemm(64)
    try:
        fn()
        sync()
        _, _, sh = xt.profile_gemm_read(shapes=True)
    finally:
        xt.profile_gemm(0)
    return [(int(r[4]), int(r[7])) for r in sh]


# ragged M (not a multiple of 256 or of 128), ragged N and K, one tile, several waves
CASES = [(256, 256, 128), (200, 96, 72), (1000, 776, 328), (64, 40, 16), (384, 512, 1024), (2048, 1536, 512)]


@pytest.mark.parametrize("c", ["f32", "bf16"])
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", CASES)
def test_pair_fwd(c, ta, tb, M, N, K, paired):
    A = synth.normal((K, M) if ta else (M, K), 140, dtype="bf16")
    B = synth.normal((N, K) if tb else (K, N), 141, dtype="bf16")
    want = O.matmul_fwd(op(A, ta), op(B, tb)) * 0.5
    C = empty((M, N), c)
    d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_c=xt.XT_F32 if c == "f32" else xt.XT_BF16, alpha=0.5)
    Ad, Bd = dev(A, "bf16"), dev(B, "bf16")
    rec = records(lambda: xt.xt_matmul_fwd(d, Ad, Bd, C))
    assert len(rec) == 1 and rec[0][0] > 1000, rec
    e = norm_err(host(C), want)
    assert e <= (1e-5 if c == "f32" else 4e-3), f"normalised error {e:.2e}"
    assert xt.device_errors() == 0


@pytest.mark.parametrize("c", ["f32", "bf16"])
def test_pair_accumulate(c, paired):
    """C += α·A@B: fp32 C through the TMA reduce-add, bf16 C through the direct stores."""
    M, N, K = 520, 264, 200
    A = synth.normal((M, K), 142, dtype="bf16")
    B = synth.normal((K, N), 143, dtype="bf16")
    C0 = synth.normal((M, N), 144, dtype=c)
    Cd = dev(C0, c)
    d = xt.matmul_desc(M, N, K, dtype_c=xt.XT_F32 if c == "f32" else xt.XT_BF16, accumulate=1)
    rec = records(lambda: xt.xt_matmul_fwd(d, dev(A, "bf16"), dev(B, "bf16"), Cd))
    assert rec[0][0] > 1000, rec
    assert norm_err(host(Cd), C0 + A @ B) <= (1e-5 if c == "f32" else 8e-3)
    assert xt.device_errors() == 0


@pytest.mark.parametrize("form", [2, 3, 4])
@pytest.mark.parametrize("c", ["f32", "bf16"])
@pytest.mark.parametrize("acc", [0, 1])
@pytest.mark.parametrize("M,N,K,ta", [(768, 768, 8192, 1), (200, 136, 8192, 1), (256, 256, 10240, 0),
                                      (1000, 776, 656, 0)])
def test_pair_split_and_stream_k(form, c, acc, M, N, K, ta, paired):
    """The paired kernel under a K split (2), stream-K over every resident pair (3) and
    lockstep K slices (4): each CTA of a pair keeps its own rows' partial; results within the
    whole-tile bound and bit-identical on a rerun; flag words left zero."""
    paired(form)
    A = synth.normal((K, M) if ta else (M, K), 145, dtype="bf16")
    B = synth.normal((K, N), 146, dtype="bf16")
    C0 = synth.normal((M, N), 147, dtype=c)
    d = xt.matmul_desc(M, N, K, trans_a=ta, dtype_c=xt.XT_F32 if c == "f32" else xt.XT_BF16, accumulate=acc,
                       alpha=0.5)
    Ad, Bd = dev(A, "bf16"), dev(B, "bf16")
    ws = xt.matmul_workspace(d)
    outs = []
    for _ in range(2):
        Cd = dev(C0, c)
        rec = records(lambda: xt.xt_matmul_fwd(d, Ad, Bd, Cd, ws=ws))
        assert len(rec) == 1 and rec[0][0] > 1000, rec
        code = rec[0][1]
        if form == 2:   # a K split (10 × splits) needs 4 k-blocks per slice: K = 656 is too short, whole tiles
            assert code == 0 if K < 1024 else code >= 20, code
        elif form == 3:
            assert code == 1000, code
        else:
            assert code > 1000, code
        outs.append(host(Cd))
    want = (C0 if acc else 0) + 0.5 * (op(A, ta) @ B)
    tol = 1e-5 if c == "f32" else (8e-3 if acc else 4e-3)
    assert norm_err(outs[0], want) <= tol
    assert np.array_equal(outs[0], outs[1]), "paired schedule is not deterministic"
    assert xt.device_errors() == 0
    assert int(ws[:4096].count_nonzero()) == 0


@pytest.mark.parametrize("M,N,K,ta,tb", [(8192, 3072, 768, 0, 0), (8192, 768, 3072, 0, 1), (8192, 2304, 768, 0, 0),
                                         (768, 3072, 8192, 1, 0), (8192, 50304, 768, 0, 1)])
def test_pair_full_size_sampled(M, N, K, ta, tb, paired):
    """The 12-layer stack's GEMM shapes on the paired kernel, sampled rows (including both
    CTAs' halves of a 256-row tile and the last row) against the oracle's product of those rows."""
    A = synth.normal((K, M) if ta else (M, K), 148, std=0.5, dtype="bf16")
    B = synth.normal((N, K) if tb else (K, N), 149, std=0.02, dtype="bf16")
    Cm = empty((M, N), "bf16")
    d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_c=xt.XT_BF16)
    Ad, Bd = dev(A, "bf16"), dev(B, "bf16")
    rec = records(lambda: xt.xt_matmul_fwd(d, Ad, Bd, Cm))
    assert len(rec) == 1 and rec[0][0] > 1000, rec
    rows = np.random.default_rng(2).choice(M, 24, replace=False)
    rows = np.concatenate([rows, [0, 127, 128, 255, 256, M - 1]])
    want = op(A, ta)[rows] @ op(B, tb)
    assert norm_err(host(Cm[torch.tensor(rows, device="cuda")]), want) <= 4e-3
    assert xt.device_errors() == 0


def test_pair_matches_single():
    """The same problem on the single-CTA and the paired kernel: both within the bound of the
    oracle, and within fp32 accumulation-order rounding of each other."""
    M, N, K = 1024, 1024, 2048
    A = synth.normal((M, K), 150, dtype="bf16")
    B = synth.normal((K, N), 151, dtype="bf16")
    d = xt.matmul_desc(M, N, K)
    Ad, Bd = dev(A, "bf16"), dev(B, "bf16")
    outs = {}
    try:
        for mode in (1, 2):
            xt.gemm_set_pairing(mode)
            C = empty((M, N))
            rec = records(lambda: xt.xt_matmul_fwd(d, Ad, Bd, C))
            assert (rec[0][0] > 1000) == (mode == 2), rec
            outs[mode] = host(C)
    finally:
        xt.gemm_set_pairing(0)
    want = A @ B
    for m in (1, 2):
        assert norm_err(outs[m], want) <= 1e-5
    assert norm_err(outs[1], outs[2]) <= 1e-5


def test_gemm_set_pairing_rejects():
    with pytest.raises(xt.XtError):
        xt.gemm_set_pairing(4)


@pytest.fixture
def multicast():
    """Forces the multicast form of the paired kernel for one test; restores the model's choice."""
    xt.gemm_set_pairing(3)
    yield
    xt.gemm_set_pairing(0)


# even numbers of 256-row tiles (a cluster's two pairs take vertically adjacent tiles): one
# tile group, ragged M / N / K (the out-of-range rows of a multicast half arrive zero-filled),
# several groups per cluster
MC_CASES = [(512, 256, 128), (384, 264, 72), (1000, 776, 328), (2048, 1536, 520), (4096, 2304, 768)]


@pytest.mark.parametrize("c", ["f32", "bf16"])
@pytest.mark.parametrize("ta,tb", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", MC_CASES)
def test_pair_multicast_fwd(c, ta, tb, M, N, K, multicast):
    """Clusters of two pairs sharing B by TMA multicast, every operand majorness, against the
    oracle with the whole-tile bounds; the launch record shows the multicast form ran."""
    A = synth.normal((K, M) if ta else (M, K), 160, dtype="bf16")
    B = synth.normal((N, K) if tb else (K, N), 161, dtype="bf16")
    want = O.matmul_fwd(op(A, ta), op(B, tb)) * 0.5
    C = empty((M, N), c)
    d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_c=xt.XT_F32 if c == "f32" else xt.XT_BF16, alpha=0.5)
    rec = records(lambda: xt.xt_matmul_fwd(d, dev(A, "bf16"), dev(B, "bf16"), C))
    assert len(rec) == 1 and rec[0][0] == 2256, rec
    e = norm_err(host(C), want)
    assert e <= (1e-5 if c == "f32" else 4e-3), f"normalised error {e:.2e}"
    assert xt.device_errors() == 0


@pytest.mark.parametrize("c", ["f32", "bf16"])
def test_pair_multicast_accumulate(c, multicast):
    """C += A@B on the multicast form: fp32 C through the TMA reduce-add, bf16 C direct."""
    M, N, K = 1024, 520, 200
    A = synth.normal((M, K), 162, dtype="bf16")
    B = synth.normal((K, N), 163, dtype="bf16")
    C0 = synth.normal((M, N), 164, dtype=c)
    Cd = dev(C0, c)
    d = xt.matmul_desc(M, N, K, dtype_c=xt.XT_F32 if c == "f32" else xt.XT_BF16, accumulate=1)
    rec = records(lambda: xt.xt_matmul_fwd(d, dev(A, "bf16"), dev(B, "bf16"), Cd))
    assert rec[0][0] == 2256, rec
    assert norm_err(host(Cd), C0 + A @ B) <= (1e-5 if c == "f32" else 8e-3)
    assert xt.device_errors() == 0


@pytest.mark.parametrize("tb", [0, 1])
def test_pair_multicast_matches_pair(tb):
    """The multicast form runs the same MMAs in the same K order on the same tiles as the plain
    pairs: bit-identical results, and identical on a rerun."""
    M, N, K = 2048, 1280, 1000
    A = synth.normal((M, K), 165, dtype="bf16")
    B = synth.normal((N, K) if tb else (K, N), 166, dtype="bf16")
    d = xt.matmul_desc(M, N, K, trans_b=tb)
    Ad, Bd = dev(A, "bf16"), dev(B, "bf16")
    outs = []
    try:
        xt.gemm_set_tile(256)
        for mode, code in ((2, 1256), (3, 2256), (3, 2256)):
            xt.gemm_set_pairing(mode)
            C = empty((M, N))
            rec = records(lambda: xt.xt_matmul_fwd(d, Ad, Bd, C))
            assert rec[0][0] == code, rec
            outs.append(host(C))
    finally:
        xt.gemm_set_pairing(0)
        xt.gemm_set_tile(0)
    assert norm_err(outs[0], A @ op(B, tb)) <= 1e-5
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    assert xt.device_errors() == 0


def test_pair_multicast_needs_even_tile_rows(multicast):
    """An odd number of 256-row tiles leaves the second pair of a cluster without a tile: the
    plain pairs run instead."""
    M, N, K = 768, 512, 256
    A = synth.normal((M, K), 167, dtype="bf16")
    B = synth.normal((K, N), 168, dtype="bf16")
    C = empty((M, N))
    d = xt.matmul_desc(M, N, K)
    rec = records(lambda: xt.xt_matmul_fwd(d, dev(A, "bf16"), dev(B, "bf16"), C))
    assert 1000 < rec[0][0] < 2000, rec
    assert norm_err(host(C), A @ B) <= 1e-5


@pytest.mark.parametrize("M,N,K,ta,tb", [(8192, 3072, 768, 0, 0), (8192, 3072, 768, 0, 1), (8192, 768, 3072, 0, 1),
                                         (8192, 2304, 768, 0, 0), (8192, 50304, 768, 0, 1)])
def test_pair_multicast_full_size_sampled(M, N, K, ta, tb, multicast):
    """The stack's 8192-row GEMM shapes on the multicast form, sampled rows (both pairs' tiles of
    a group, both CTAs' halves of a tile, the last row) against the oracle's product of those rows."""
    A = synth.normal((K, M) if ta else (M, K), 169, std=0.5, dtype="bf16")
    B = synth.normal((N, K) if tb else (K, N), 170, std=0.02, dtype="bf16")
    Cm = empty((M, N), "bf16")
    d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=tb, dtype_c=xt.XT_BF16)
    rec = records(lambda: xt.xt_matmul_fwd(d, dev(A, "bf16"), dev(B, "bf16"), Cm))
    assert len(rec) == 1 and rec[0][0] == 2256, rec
    rows = np.random.default_rng(3).choice(M, 24, replace=False)
    rows = np.concatenate([rows, [0, 127, 128, 255, 256, 383, 384, 511, M - 1]])
    want = op(A, ta)[rows] @ op(B, tb)
    assert norm_err(host(Cm[torch.tensor(rows, device="cuda")]), want) <= 4e-3
    assert xt.device_errors() == 0


@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("M,N,K", [(1000, 776, 328), (8192, 768, 3072), (256, 192, 64)])
def test_pair_tile_192(ta, M, N, K, paired):
    """Paired 256 × 192 tiles (96 rows of B per CTA), offered for K-major B only."""
    xt.gemm_set_tile(192)
    try:
        A = synth.normal((K, M) if ta else (M, K), 152, dtype="bf16")
        B = synth.normal((N, K), 153, dtype="bf16")   # [N, K]: K-major
        C = empty((M, N))
        d = xt.matmul_desc(M, N, K, trans_a=ta, trans_b=1)
        rec = records(lambda: xt.xt_matmul_fwd(d, dev(A, "bf16"), dev(B, "bf16"), C))
        assert rec[0][0] == 1192, rec
        assert norm_err(host(C), op(A, ta) @ B.T) <= 1e-5
        assert xt.device_errors() == 0
    finally:
        xt.gemm_set_tile(0)


def test_gemm_set_tile_rejects():
    with pytest.raises(xt.XtError):
        xt.gemm_set_tile(96)
