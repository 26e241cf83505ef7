"""mfsdp_gemm_f32_batched (the 3xTF32 tcgen05 GEMM behind the second-order optimizers)
against the fp64 product of the same fp32 inputs.

Cases: every transpose combination; one launch holding problems of different shapes; ragged
sizes (m, n, k not multiples of the 128 x 256 x 32 tiles, k = 1, a 1 x 1 problem); pitches
larger than the row (and not multiples of 4, so the loads fall back from 16-byte vectors);
alpha / beta with C read back; an empty problem in the table; both operands K-major with
TMA-addressable pitches (the launch's TMA variant).  Bound: the 3xTF32 error is
below 2^-21 of each product |a||b|, so |C - C_ref| <= k 2^-20 max|a| max|b| elementwise and
the relative Frobenius error stays under 2e-6 (an fp32 FFMA GEMM of these sizes is ~1e-6).
A plain TF32 product (2^-11) fails both.
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _mat(rows, cols, pitch, gen, dev, scale=1.0):
    base = torch.randn(rows, pitch, generator=gen, device=dev) * scale
    return base[:, :cols]


def _ref(a, b, c0, alpha, beta, ta, tb):
    A = a.double().cpu().numpy()
    B = b.double().cpu().numpy()
    A = A.T if ta else A
    B = B.T if tb else B
    return alpha * (A @ B) + beta * c0.double().cpu().numpy()


def _run(shapes, ta, tb, alpha=1.0, beta=0.0, pitch_extra=0, seed=0):
    from matrix_optimizer_owner_gb300 import mfsdp
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    probs, refs = [], []
    for (m, n, k) in shapes:
        a = _mat(k, m, m + pitch_extra, gen, dev) if ta else _mat(m, k, k + pitch_extra, gen, dev)
        b = _mat(n, k, k + pitch_extra, gen, dev) if tb else _mat(k, n, n + pitch_extra, gen, dev)
        c = _mat(m, n, n + pitch_extra, gen, dev)
        refs.append((_ref(a, b, c, alpha, beta, ta, tb), a, b, k))
        probs.append((a, b, c, alpha, beta))
    mfsdp.mfsdp_gemm_f32_batched(probs, ta, tb)
    torch.cuda.synchronize()
    assert mfsdp.mfsdp_query_status() == 0
    for (ref, a, b, k), (_, _, c, _, _) in zip(refs, probs):
        got = c.double().cpu().numpy()
        if ref.size == 0:
            continue
        bound = max(k, 1) * 2.0 ** -20 * float(a.abs().max()) * float(b.abs().max()) * abs(alpha)
        err = np.abs(got - ref)
        assert err.max() <= bound + 1e-7 * np.abs(ref).max(), (shapes, ta, tb, err.max(), bound)
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= 2e-6, (shapes, ta, tb, rel)


@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("tb", [0, 1])
def test_transposes_and_mixed_batch(ta, tb):
    _run([(300, 520, 700), (128, 256, 32), (1, 1, 1), (257, 129, 65), (768, 768, 768)], ta, tb,
         seed=ta * 2 + tb)


def test_k_major_operands_by_tma():
    # both operands K-major with pitches a multiple of 4 floats: the launch takes the TMA
    # variant (every problem qualifies); ragged m, n and k, alpha and beta
    _run([(300, 520, 700), (128, 256, 32), (257, 129, 68), (768, 768, 768), (130, 70, 4),
          (1, 300, 36)], 0, 1, alpha=0.7, beta=0.3, seed=11)


def test_tma_launches_split_at_64_problems():
    # 70 TMA-eligible problems: the launch carries the tensor maps of at most 64, so the
    # table runs as two launches (64 + 6), longest contraction first
    shapes = [(32 + 8 * (i % 5), 40 + 16 * (i % 3), 36 + 4 * (i % 7)) for i in range(70)]
    _run(shapes, 0, 1, alpha=1.0, beta=0.5, seed=12)


def test_alpha_beta_and_ragged_pitches():
    _run([(200, 300, 97), (64, 1000, 3), (130, 70, 1)], 0, 1, alpha=0.05, beta=0.95,
         pitch_extra=3, seed=7)
    _run([(200, 300, 97), (33, 17, 501)], 1, 0, alpha=-1.5, beta=2.0, pitch_extra=5, seed=8)


def test_statistics_shapes_of_a_transformer_layer():
    # G G^T and G^T G of the four GPT-2-small layer matrices, in the two launches the
    # optimizers issue (L sides: A = G, B = G^T; R sides: A = G^T, B = G)
    shapes = [(2304, 768), (768, 768), (3072, 768), (768, 3072)]
    _run([(r, r, c) for r, c in shapes], 0, 1, alpha=0.05, beta=0.95, seed=9)
    _run([(c, c, r) for r, c in shapes], 1, 0, alpha=0.05, beta=0.95, seed=10)


def test_empty_problems_are_no_work():
    from matrix_optimizer_owner_gb300 import mfsdp
    dev = torch.device("cuda", 0)
    a = torch.ones(4, 0, device=dev)
    b = torch.ones(0, 5, device=dev)
    c = torch.full((4, 5), 3.0, device=dev)
    # k = 0: C = alpha * 0 + beta * C
    mfsdp.mfsdp_gemm_f32_batched([(a, b, c, 1.0, 0.5)])
    torch.cuda.synchronize()
    assert torch.all(c == 1.5)
    e = torch.empty(0, 5, device=dev)
    mfsdp.mfsdp_gemm_f32_batched([(e, torch.ones(5, 5, device=dev), torch.empty(0, 5, device=dev),
                                   1.0, 0.0)])
    torch.cuda.synchronize()
    assert mfsdp.mfsdp_query_status() == 0
