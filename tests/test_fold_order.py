"""The order in which split partials are folded decides output bits.

"P3: native paged-KV continuous-batching sampler", Design / paged.py asks for a fixed KV split
per context length and no atomics, so that a row's bits do not depend on the batch. The split
combine of this library folds a row's splits in ascending order with the scalar,
round-to-nearest fp32 operations below (the combine kernel and the in-kernel fold of prefill
tiles use exactly these, in this order):

    M' = max(M, m_s)
    a  = 2^((M - M') c)    (1 when M == M')
    b  = 2^((m_s - M') c)  (1 when m_s == M')
    L  = L a + l_s b
    ACC = ACC a + acc_s b
    out = bf16(ACC * rcp(L))

This test restates that fold on the CPU in float32 (numpy rounds every float32 operation to
nearest and never fuses a multiply-add; its exp2 is not the GPU's ex2.approx, which does not
matter for the point made here) and shows, on the decode workload's multi-split rows, that
folding the same partials in descending order changes output bits. An order chosen at run
time, as atomics would choose it, therefore could not give batch-invariant bits; the fixed
ascending order can."""
import numpy as np

from continuous_batching_gb300 import workloads as wl

SPLIT = 2048
C = np.float32(np.log2(np.e) / np.sqrt(128.0))


def _bf16(x):
    return wl.f32_to_bf16_bits(np.asarray(x, np.float32))


def _fold(partials, rounded=True):
    """partials: list of (m float32, l float32, acc float32[D]) in the order to fold. Returns
    the bf16 output bits, or (rounded=False) the fp32 value before that rounding."""
    M, L, A = partials[0]
    M, L, A = np.float32(M), np.float32(L), A.astype(np.float32).copy()
    for m, l, acc in partials[1:]:
        mn = np.float32(max(M, m))
        a = np.float32(1) if M == mn else np.exp2(np.float32(np.float32(M - mn) * C))
        b = np.float32(1) if m == mn else np.exp2(np.float32(np.float32(m - mn) * C))
        L = np.float32(np.float32(L * a) + np.float32(l * b))
        A = (A * a).astype(np.float32) + (acc * b).astype(np.float32)
        M = mn
    inv = np.float32(np.float32(1) / L)
    return _bf16(A * inv) if rounded else (A * inv).astype(np.float32)


def _partials(q, K, V):
    """Per split: (m = max raw score, l = sum of 2^((s - m) c), acc = sum of p v) in float32,
    from bf16-valued q, K, V of one head."""
    out = []
    s_all = (K @ q).astype(np.float32)
    for lo in range(0, K.shape[0], SPLIT):
        s = s_all[lo:lo + SPLIT]
        m = np.float32(s.max())
        p = np.exp2((s - m).astype(np.float32) * C).astype(np.float32)
        out.append((m, np.float32(p.sum(dtype=np.float32)),
                    (p[:, None] * V[lo:lo + SPLIT]).sum(axis=0, dtype=np.float32)))
    return out


def test_descending_fold_changes_bits_on_decode_rows():
    st = wl.make_config("decode", with_pool=False)
    long_ctx = [int(c) for c in st.ctx_lens if c > SPLIT]
    assert len(long_ctx) >= 10
    rng = np.random.default_rng(17)
    differ = differ32 = total = 0
    bits = lambda shape: wl.random_bf16(rng, shape).astype(np.uint32) << 16
    for ctx in long_ctx:
        K = bits((ctx, 128)).view(np.float32)           # one KV head and its 4 query heads
        V = bits((ctx, 128)).view(np.float32)
        for h in range(4):
            q = bits((128,)).view(np.float32)
            parts = _partials(q, K, V)
            up, down = _fold(parts), _fold(parts[::-1])
            differ += int((up != down).sum())
            differ32 += int((_fold(parts, False) != _fold(parts[::-1], False)).sum())
            total += up.size
            # both orders are the same softmax up to rounding
            ref = np.exp((K @ q).astype(np.float64) * (C / np.log2(np.e)))
            ref = (ref / ref.sum()) @ V.astype(np.float64)
            got = (up.astype(np.uint32) << 16).view(np.float32)
            assert np.abs(got - ref).max() <= 2.0 ** -5 * np.sqrt((ref ** 2).mean()) + 1e-4
    print(f"fp32 results differing: {differ32} of {total}; bf16 outputs differing: {differ}")
    assert differ32 > total // 10, "the fold order barely changed the fp32 results"
    assert differ > 0, "ascending and descending folds gave the same output bits everywhere"
    assert differ < total
