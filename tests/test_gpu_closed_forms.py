"""Closed forms of causal softmax attention run through the CUDA path at long context, where
the absolute tolerance alone could not see a missing key tile or split.

- Dominant key: when one key's score exceeds every other by far more than the exponent range
  (here by about 86 in natural-log units), softmax puts all the weight on it and the output
  row is that key's V row. Such a key is planted in the first, a middle and the last 128-key
  tile of every 2048-key split, at ctx 16,384 and 40,960, for decode rows and for 512-row
  prefill chunks. A kernel that skipped any of those tiles or splits returns an average of
  random rows instead of the planted V row.
- Identical keys: all scores are equal, so the output is the mean of V over the row's keys.
- Causal boundary: a dominant key inside a prefill chunk is seen by the rows at or after its
  position and by no row before it.

The definition being checked is "P3: native paged-KV continuous-batching sampler",
Design / paged.py ('row' mode: each query row attends exactly its own keys) with the GQA map
of Tensor parallelism / Design; the closed forms follow from the softmax itself.
"""
import numpy as np
import pytest

import oracle.paged_attention as pa
from continuous_batching_gb300 import workloads as wl
from tests.gpu_util import assert_close, run_step

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

SPLIT, TILE = 2048, 128
ONE, MINUS_ONE, EIGHT, MINUS_EIGHT = 0x3F80, 0xBF80, 0x4100, 0xC100   # bf16 bit patterns


@pytest.fixture(scope="module", autouse=True)
def lib():
    from continuous_batching_gb300 import build
    from continuous_batching_gb300 import binding as bd
    build.build()
    return bd.load()


def hadamard(n):
    h = np.array([[1]], np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def _key_ref(st, s, pos):
    """Where K/V of position pos of sequence s lives: ('new', token) or ('pool', block, off)."""
    ctx, nq = int(st.ctx_lens[s]), int(st.n_q[s])
    if pos >= ctx - nq:
        return ("new", int(st.cu_seqlens_q[s]) + pos - (ctx - nq))
    return ("pool", int(st.block_table[s, pos // st.block_size]), pos % st.block_size)


def _set_k(st, s, pos, kvh, bits):
    r = _key_ref(st, s, pos)
    if r[0] == "new":
        st.k_new[r[1], kvh] = bits
    else:
        st.k_pool[r[1], r[2], kvh] = bits


def _get_v(st, s, pos, kvh):
    r = _key_ref(st, s, pos)
    return st.v_new[r[1], kvh] if r[0] == "new" else st.v_pool[r[1], r[2], kvh]


def _split_positions(ctx, limit, rng):
    """A key in the first, a middle and the last tile of every split of [0, ctx), each below
    limit (positions past it are moved into the last tile before it)."""
    out = []
    for sp in range((ctx + SPLIT - 1) // SPLIT):
        base = sp * SPLIT
        n_tiles = min(SPLIT, ctx - base + TILE - 1) // TILE
        for t in (0, n_tiles // 2, n_tiles - 1):
            p = base + t * TILE + int(rng.integers(0, TILE))
            if p >= limit:
                p = limit - 1 - int(rng.integers(0, TILE))
            out.append(p)
    return out


def _plant_dominant(st, seqs, positions, rng):
    """Each (sequence, KV head, head-in-group) of `seqs` gets its own direction u (rows of a
    Hadamard matrix, orthogonal within a KV head): its q rows are u and one key at a planted
    position is 8 u, every other key stays N(0, 1). Positions are dealt from `positions` in
    order (then at random). Returns {(s, head): position}."""
    H = hadamard(st.D)
    g = st.Hq // st.Hkv
    plan = {}
    it = iter(positions)
    for s in seqs:
        a, b = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        lo = int(st.ctx_lens[s]) - (b - a)
        for kvh in range(st.Hkv):
            used = set()
            for j in range(g):
                p = next(it, None)
                while p is None or p in used:
                    p = int(rng.integers(0, lo if b - a > 1 else int(st.ctx_lens[s])))
                used.add(p)
                u = H[1 + j]
                h = kvh * g + j
                st.q[a:b, h] = np.where(u > 0, ONE, MINUS_ONE).astype(np.uint16)
                _set_k(st, s, p, kvh, np.where(u > 0, EIGHT, MINUS_EIGHT).astype(np.uint16))
                plan[(s, h)] = p
    return plan


def _check_dominant(st, out, plan):
    got = pa.bf16_to_f64(out)
    g = st.Hq // st.Hkv
    bad = []
    for (s, h), p in plan.items():
        a, b = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        want = pa.bf16_to_f64(_get_v(st, s, p, h // g))
        d = np.abs(got[a:b, h] - want[None, :])
        # the planted V row to within one bf16 unit in the last place
        if not np.all(d <= 2.0 ** -7 * np.abs(want)[None, :] + 1e-30):
            bad.append((s, h, p, float(d.max())))
    assert not bad, f"{len(bad)} (sequence, head) pairs miss their dominant key: {bad[:6]}"


def test_dominant_key_in_every_split_at_16k_and_40k():
    rng = np.random.default_rng(2024)
    ctx = [16384, 40960, 40960, 16384, 40960, 40960]
    n_q = [1, 1, 1, 512, 512, 512]
    st = wl.make_step(32, 8, 128, 16, ctx, n_q, seed=91)
    plan = {}
    # decode rows: the planted keys cover every split; one lands on the token written in
    # this very step (the row's own position)
    p16 = _split_positions(16384, 16384, rng) + [16383]
    p40 = _split_positions(40960, 40960, rng) + [40959]
    plan.update(_plant_dominant(st, [0], p16, rng))
    plan.update(_plant_dominant(st, [1, 2], p40, rng))
    # prefill chunks (512 rows at prior offset ctx - 512): keys below the chunk, so that
    # every row of the chunk sees its head's planted key
    plan.update(_plant_dominant(st, [3], _split_positions(16384, 16384 - 512, rng), rng))
    plan.update(_plant_dominant(st, [4, 5], _split_positions(40960, 40960 - 512, rng), rng))
    covered = {p // TILE for (s, h), p in plan.items() if s in (1, 2)}
    assert all(sp * 16 in covered and sp * 16 + 15 in covered for sp in range(20))
    out, kp, vp, err = run_step(st, torch)
    assert err == 0
    _check_dominant(st, out, plan)


def test_identical_keys_give_the_mean_of_v():
    """All keys of a (sequence, KV head) equal: uniform weights over keys 0..p, so row p's
    output is the mean of V[0..p]; decode rows and 512-row prefill chunks at 16k and 40k."""
    rng = np.random.default_rng(7)
    ctx = [16384, 40960, 16384, 40960]
    n_q = [1, 1, 512, 512]
    st = wl.make_step(32, 8, 128, 16, ctx, n_q, seed=92)
    g = st.Hq // st.Hkv
    for s in range(st.B):
        k0 = wl.random_bf16(rng, (st.Hkv, st.D))
        L = int(st.ctx_lens[s])
        nblk = (L + st.block_size - 1) // st.block_size
        st.k_pool[st.block_table[s, :nblk]] = k0[None, None]
        a, b = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        st.k_new[a:b] = k0[None]
    out, kp, vp, err = run_step(st, torch)
    assert err == 0
    got = pa.bf16_to_f64(out)
    vpool = pa.bf16_to_f64(vp.view(torch.int16).cpu().numpy().view(np.uint16))
    for s in range(st.B):
        L = int(st.ctx_lens[s])
        V = pa.gather(vpool, st.block_table[s], L)                 # [Hkv, L, D]
        cm = np.cumsum(V, axis=1) / np.arange(1, L + 1)[None, :, None]
        a, b = int(st.cu_seqlens_q[s]), int(st.cu_seqlens_q[s + 1])
        pos = L - (b - a) + np.arange(b - a)
        want = cm[np.arange(st.Hq) // g][:, pos].transpose(1, 0, 2)  # [rows, Hq, D]
        d = np.abs(got[a:b] - want)
        # bf16 rounding of the mean plus the fp32 sum of up to 40,960 terms
        ok = d <= 2.0 ** -7 * np.abs(want) + 4e-6
        assert np.all(ok), (f"sequence {s}: {int((~ok).sum())} elements off the mean, "
                            f"max |diff| {d.max():.3e}")


def test_causal_boundary_inside_a_prefill_chunk():
    """A dominant key at position j inside a 512-row chunk (in this step's own new keys):
    rows at j or later return its V row; the rows before j do not see it and match the
    oracle."""
    rng = np.random.default_rng(11)
    st = wl.make_step(32, 8, 128, 16, [3000, 2100], [512, 1], seed=93)
    off = 3000 - 512
    H = hadamard(st.D)
    g = st.Hq // st.Hkv
    j = off + 37
    for kvh in range(st.Hkv):
        u = H[1 + kvh]
        st.q[0:512, kvh * g:(kvh + 1) * g] = np.where(u > 0, ONE, MINUS_ONE).astype(np.uint16)[None, None]
        _set_k(st, 0, j, kvh, np.where(u > 0, EIGHT, MINUS_EIGHT).astype(np.uint16))
    out, kp, vp, err = run_step(st, torch)
    assert err == 0
    got = pa.bf16_to_f64(out)
    for kvh in range(st.Hkv):
        want = pa.bf16_to_f64(_get_v(st, 0, j, kvh))
        d = np.abs(got[37:512, kvh * g:(kvh + 1) * g] - want[None, None])
        assert np.all(d <= 2.0 ** -7 * np.abs(want)[None, None] + 1e-30), f"kv head {kvh}"
    rows = np.arange(0, 37)
    ref = pa.attention_rows(st.q, kp.view(torch.int16).cpu().numpy().view(np.uint16),
                            vp.view(torch.int16).cpu().numpy().view(np.uint16), st.block_table,
                            st.cu_seqlens_q, st.ctx_lens, st.Hq, rows)
    assert_close(out[rows], ref, "rows before the planted key")
    # those rows really do differ from the planted V row (the check above has teeth)
    far = np.abs(got[rows][:, 0] - pa.bf16_to_f64(_get_v(st, 0, j, 0))[None]).max(axis=-1)
    assert far.min() > 0.1
