"""Pins of the oracle's expert-parallel MoE reference (FP8 dispatch, BF16
combine: "Six Reasons Deepseek Ai Is A Waste Of Time", para. 4) and of its
BF16 rounding (CPU only).

bf16_round: equal to torch's FP32 -> BF16 conversion (round to nearest even)
on FP32 inputs, every midpoint between BF16 neighbours goes to the even one,
and BF16 values are fixed points.
moe_ep_reference: an exact closed form with two experts and gate weights;
permuting the expert labels changes nothing; two experts with the same
weights and gates summing to one give the single-expert result; doubling
every gate doubles the output; and a brute-force evaluation written from the
definition (decode, scale, dot product per token and expert) on a tiny case."""
import numpy as np
import torch

import fp8q_inputs as fi


def test_bf16_round_matches_torch_and_ties_to_even(oracle):
    x = (np.random.default_rng(0).standard_normal(200000) * 37.0).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(oracle.bf16_round(x.astype(np.float64)), ref)
    # 1 + k/128 are consecutive BF16 values in [1, 2); their midpoints go to
    # the neighbour with an even last mantissa bit
    k = np.arange(128)
    mid = 1.0 + (k + 0.5) / 128.0
    want = np.where(k % 2 == 0, 1.0 + k / 128.0, 1.0 + (k + 1) / 128.0)
    assert np.array_equal(oracle.bf16_round(mid), want)
    assert np.array_equal(oracle.bf16_round(-mid), -want)
    vals = 1.0 + k / 128.0
    assert np.array_equal(oracle.bf16_round(vals * 2.0 ** 20), vals * 2.0 ** 20)
    assert oracle.bf16_round(0.0) == 0.0


def quant_experts(oracle, W):
    E, N, H = W.shape
    W8 = np.empty((E, N, H), np.uint8)
    sW = np.empty((E, N // 128, H // 128), np.float32)
    for e in range(E):
        W8[e], sW[e] = oracle.quant_128x128(W[e])
    return W8, sW


def test_moe_closed_form(oracle):
    """Activations all 7 and expert weights all -7/16 or 7/8: every scale is a
    power of two and every byte 448, so y = 256 * 7 * w exactly; the gates
    0.5 and 0.25 give out = 0.5 y_a + 0.25 y_b, BF16-exact here."""
    T, H, N = 4, 256, 128
    x = np.full((T, H), 7.0, np.float32)
    W = np.stack([np.full((N, H), -0.4375, np.float32), np.full((N, H), 0.875, np.float32)])
    W8, sW = quant_experts(oracle, W)
    ids = np.array([[0, 1]] * T)
    gates = np.array([[0.5, 0.25]] * T, np.float32)
    out, y, _ = oracle.moe_ep_reference(x, ids, gates, W8, sW)
    ya, yb = 256 * 7 * -0.4375, 256 * 7 * 0.875
    assert np.all(y[:, 0] == ya) and np.all(y[:, 1] == yb)
    assert np.all(out == 0.5 * ya + 0.25 * yb)


def random_case(T=32, H=256, N=256, E=6, k=3, seed=5):
    rng = np.random.default_rng(seed)
    x = fi.gaussian((T, H), fi.rng_for(seed, 0), 1.0, 0.01, 30.0)
    W = fi.gaussian((E, N, H), fi.rng_for(seed, 1), 0.02, bf16=False)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
    gates = rng.random((T, k)).astype(np.float32)
    return x, W, ids, gates


def test_moe_invariances(oracle):
    x, W, ids, gates = random_case()
    W8, sW = quant_experts(oracle, W)
    out, _, _ = oracle.moe_ep_reference(x, ids, gates, W8, sW)
    # relabel the experts
    perm = np.array([3, 0, 5, 1, 4, 2])              # new label of old expert e is perm[e]
    inv = np.argsort(perm)
    out_p, _, _ = oracle.moe_ep_reference(x, perm[ids], gates, W8[inv], sW[inv])
    assert np.array_equal(out, out_p)
    # doubling every gate doubles the output exactly
    out2, _, _ = oracle.moe_ep_reference(x, ids, gates * 2, W8, sW)
    assert np.array_equal(out2, 2 * out)
    # two experts with the same weights, gates 1/2 and 1/2: the single result
    W8d = np.concatenate([W8[:1], W8[:1]])
    sWd = np.concatenate([sW[:1], sW[:1]])
    T = x.shape[0]
    outd, y, _ = oracle.moe_ep_reference(x, np.array([[0, 1]] * T), np.full((T, 2), 0.5, np.float32),
                                         W8d, sWd)
    assert np.array_equal(outd, oracle.bf16_round(y[:, 0]))


def test_moe_brute_force_tiny(oracle):
    """The definition written out with numpy only: decode every byte, apply
    the tile and block scales, dot products in FP64, BF16 rounding of each
    expert result, gate-weighted sum, BF16 rounding."""
    x, W, ids, gates = random_case(T=6, H=256, N=128, E=4, k=2, seed=9)
    W8, sW = quant_experts(oracle, W)
    out, _, _ = oracle.moe_ep_reference(x, ids, gates, W8, sW)
    q, s = oracle.quant_1x128(x)
    xa = oracle.e4m3_decode(q) * np.repeat(s.T.astype(np.float64), 128, axis=1)
    want = np.zeros_like(out)
    for t in range(x.shape[0]):
        acc = 0.0
        for j in range(ids.shape[1]):
            e = ids[t, j]
            we = oracle.e4m3_decode(W8[e]) * np.kron(sW[e].astype(np.float64), np.ones((128, 128)))
            yt = np.array([np.dot(xa[t], we[n]) for n in range(we.shape[0])])
            acc = acc + np.float64(gates[t, j]) * oracle.bf16_round(yt)
        want[t] = oracle.bf16_round(acc)
    assert np.array_equal(out, want)
