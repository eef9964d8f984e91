"""Pins of the CPU oracle to facts it does not define itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle breaks the fact.  ``test_oracle_pins.py`` runs them on the
oracle; ``test_oracle_mutations.py`` runs them on copies of the oracle with a
planted mistake and requires that some pin fails.

What pins what:
  * Philox4x32-10: Triton's library Philox (``tl.philox``, run in its CPU
    interpreter) on random counters and 64-bit keys; statistics of the stream
    ("Add stochastic rounding and philox RNG helpers", Tests: uniform and
    free of repeats).
  * element -> (counter, word) mapping: the same independent Philox on the
    counter ((i>>2) lo, (i>>2) hi, step, 0) and key (seed lo, seed hi).
  * stochastic rounding: the exhaustive closed forms of the same page's Tests
    section (over all 65,536 random values the number of round-ups equals the
    discarded low 16 bits, the two bracketing values, exact mean), Inf/NaN.
  * round-to-nearest-even: torch's float32 -> bfloat16 conversion.
  * AdamW: a textbook binary64 AdamW recurrence (Loshchilov and Hutter) and
    torch.optim.AdamW over 100 steps ("adamw-sr", Correctness: < 1e-4), plus
    special cases with closed forms (no gradient; first step; eps-dominated).
  * the sub-ULP demonstration ("adamw-sr", introduction; tests/golden).
  * shard invariance ("adamw-sr", Method and Correctness).
  * the bf16 GEMM with a stochastic-rounding epilogue ("Add stochastic
    rounding and philox RNG helpers", Consumer): exact rational sums of tiny
    non-square products (Python fractions), rounded once to binary32, then
    each element rounded with its own Philox word; closed forms where the
    product is exactly a bf16 value (one-hot rows pick elements of B; small
    integer sums), which every seed and both roundings must reproduce.
"""
import json
import os

import numpy as np

from stochastic_rounding_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def f32_from_bits(u):
    return np.asarray(u, dtype=np.uint32).view(np.float32)


def bits_from_f32(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def bf16_value(h):
    """float64 value of bf16 patterns (via torch's conversion)."""
    return W.bf16_bits_to_f32(np.asarray(h, dtype=np.uint16)).astype(np.float64)


def bf16_is_nan(h):
    h = np.asarray(h, dtype=np.uint32)
    return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)


# --------------------------------------------------------------------------
# Philox
# --------------------------------------------------------------------------

def make_philox_cases(seed=20261202):
    """Random counters/keys, plus element-mapping cases (i, step, seed)."""
    rng = np.random.default_rng(seed)
    n = 4096
    c = {k: rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
         for k in ("c0", "c1", "c2", "c3")}
    keys = rng.integers(0, 2**64 - 1, n, dtype=np.uint64, endpoint=True)
    keys[:4] = [0, 1, 2**32, 2**64 - 1]
    c["seed"] = keys
    m = 1024
    idx = rng.integers(0, 2**42, m, dtype=np.uint64)
    idx[:8] = [0, 1, 2, 3, 4, 5, 2**32 * 4 + 3, 2**34 + 6]
    steps = rng.integers(1, 2**32, m, dtype=np.uint64).astype(np.uint32)
    seeds = rng.integers(0, 2**64 - 1, m, dtype=np.uint64, endpoint=True)
    q = idx >> np.uint64(2)
    mc = dict(c0=(q & np.uint64(0xFFFFFFFF)).astype(np.uint32),
              c1=(q >> np.uint64(32)).astype(np.uint32),
              c2=steps, c3=np.zeros(m, np.uint32), seed=seeds)
    both = {k: np.concatenate([c[k], mc[k]]) for k in c}
    return dict(inputs=both, n_random=n, idx=idx, steps=steps, seeds=seeds)


def pin_philox_matches_reference(o, cases, ref_words):
    """Oracle Philox words == Triton's Philox words on random counters/keys."""
    d = cases["inputs"]
    n = cases["n_random"]
    got = np.empty((n, 4), dtype=np.uint32)
    for j in range(n):
        s = int(d["seed"][j])
        got[j] = o.philox4x32_10([d["c0"][j], d["c1"][j], d["c2"][j], d["c3"][j]],
                                 [s & 0xFFFFFFFF, s >> 32])
    bad = np.nonzero((got != ref_words[:n]).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} of {n} Philox blocks differ from the reference; first {bad[:4]}"


def pin_element_mapping(o, cases, ref_words):
    """Element i at (seed, step) draws word i&3 of Philox(((i>>2) lo, hi, step, 0))."""
    n = cases["n_random"]
    ref = ref_words[n:]
    for j, (i, st, sd) in enumerate(zip(cases["idx"], cases["steps"], cases["seeds"])):
        want = int(ref[j][int(i) & 3])
        got = o.element_word(int(i), int(st), int(sd))
        assert got == want, f"element {int(i)} step {int(st)} seed {int(sd)}: {got:#x} != {want:#x}"


def pin_philox_fill_layout(o, cases, ref_words):
    """philox_fill(n, base, c2, c3, seed) row j == Philox((base+j) lo, hi, c2, c3)."""
    d = cases["inputs"]
    for j in range(0, 64):
        s = int(d["seed"][j])
        base = int(d["c0"][j]) | (int(d["c1"][j]) << 32)
        rows = o.philox_fill(1, base, int(d["c2"][j]), int(d["c3"][j]), s)
        assert (rows[0] == ref_words[j]).all(), f"fill row differs at case {j}"
    # a run crossing a 2^32 boundary of the low counter word carries into word 1
    base = (7 << 32) + 0xFFFFFFFE
    rows = o.philox_fill(4, base, 5, 9, 77)
    for j in range(4):
        c = base + j
        want = o.philox4x32_10([c & 0xFFFFFFFF, c >> 32, 5, 9], [77, 0])
        assert (rows[j] == want).all(), "counter carry into the high word is wrong"


def pin_philox_statistics(o):
    """Uniform bytes / low halves / bits, birthday-rate word collisions, and
    no repeated 128-bit blocks over 2^20 consecutive counters."""
    n = 1 << 20
    w = o.philox_fill(n, 0, 3, 0, 0x0123456789ABCDEF)
    flat = w.reshape(-1)
    # bytes
    counts = np.bincount(flat.view(np.uint8), minlength=256).astype(np.float64)
    e = counts.sum() / 256
    chi = ((counts - e) ** 2 / e).sum()
    assert abs(chi - 255) < 6 * np.sqrt(2 * 255), f"byte chi2 {chi:.1f}"
    # low 16 bits (the bits stochastic rounding uses)
    lows = (flat & 0xFFFF).astype(np.int64)
    counts = np.bincount(lows, minlength=65536).astype(np.float64)
    e = counts.sum() / 65536
    chi = ((counts - e) ** 2 / e).sum()
    assert abs(chi - 65535) < 6 * np.sqrt(2 * 65535), f"low-16 chi2 {chi:.1f}"
    # each bit position
    bits = np.unpackbits(flat.view(np.uint8)).reshape(-1, 32).sum(axis=0)
    half = flat.size / 2
    assert np.all(np.abs(bits - half) < 6 * np.sqrt(flat.size) / 2), "biased bit position"
    # collisions of word 0 at the birthday rate; 128-bit blocks all distinct
    w0 = np.sort(w[:, 0])
    coll = int((w0[1:] == w0[:-1]).sum())
    expect = n * (n - 1) / 2 / 2**32
    assert abs(coll - expect) < 6 * np.sqrt(expect), f"word-0 collisions {coll} vs {expect:.0f}"
    blocks = np.unique(w.view(np.dtype((np.void, 16))))
    assert blocks.size == n, "repeated 128-bit Philox block"


# --------------------------------------------------------------------------
# Stochastic rounding / RNE
# --------------------------------------------------------------------------

def sr_edge_patterns():
    pats = [0x00000000, 0x80000000, 0x3F800000, 0xBF800000, 0x3F800001, 0x3F80FFFF,
            0x3F807FFF, 0x3F808000, 0x3F808001, 0x00000001, 0x0000FFFF, 0x00010000,
            0x807FFFFF, 0x007FFFFF, 0x00800000, 0x7F7F0000, 0x7F7EFFFF, 0x7F7F7FFF,
            0x4B800001, 0xC0490FDB, 0x3DCCCCCD, 0x33D6BF95]
    return np.array(pats, dtype=np.uint32)


def pin_sr_exhaustive(o, n_random=1500, seed=11):
    """Over all 65,536 values of the low random half: out is one of the two
    bracketing bf16 values; exactly low16(x) of them round up, namely those
    with r >= 65536 - low16(x); the high random half is ignored; the mean of
    the outputs equals x exactly (in binary64, where it is finite)."""
    rng = np.random.default_rng(seed)
    rand = rng.integers(0, 2**32, n_random, dtype=np.uint64).astype(np.uint32)
    rand = rand[((rand & 0x7F800000) != 0x7F800000)]          # finite only
    pats = np.concatenate([sr_edge_patterns(), rand])
    r_low = np.arange(65536, dtype=np.uint32)
    hi_junk = rng.integers(0, 2**16, 65536, dtype=np.uint64).astype(np.uint32) << 16
    for u in pats:
        u = int(u)
        x = np.full(65536, f32_from_bits(np.uint32(u)), dtype=np.float32)
        out = o.sr_fill(x, 0, 1, 0, rbits=r_low | hi_junk)
        lo = u >> 16
        L = u & 0xFFFF
        assert np.all((out == lo) | (out == lo + 1)), f"{u:#010x}: output off the two bracketing values"
        ups = out == lo + 1
        assert int(ups.sum()) == L, f"{u:#010x}: {int(ups.sum())} round-ups, expected {L}"
        assert np.array_equal(ups, r_low >= 65536 - L), f"{u:#010x}: wrong set of round-ups"
        if ((lo + 1) & 0x7F80) != 0x7F80:                      # both neighbours finite
            mean = bf16_value(out).sum() / 65536.0
            xv = float(f32_from_bits(np.uint32(u)))
            assert mean == xv, f"{u:#010x}: mean {mean!r} != x {xv!r}"


def pin_sr_inf_nan(o):
    """+-Inf pass through for every random value; NaNs stay NaN (sign kept,
    quiet), also NaNs whose payload sits in the discarded low half."""
    r_all = np.arange(65536, dtype=np.uint32) * 65537
    for u in (0x7F800000, 0xFF800000):
        x = np.full(65536, f32_from_bits(np.uint32(u)), dtype=np.float32)
        out = o.sr_fill(x, 0, 1, 0, rbits=r_all)
        assert np.all(out == (u >> 16)), f"Inf {u:#x} not preserved"
    nans = [0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001, 0x7FFFFFFF, 0xFFFFFFFF,
            0x7FBFFFFF, 0x7F80FFFF, 0x7FFF8000, 0x7FA00000]
    for u in nans:
        x = np.full(65536, f32_from_bits(np.uint32(u)), dtype=np.float32)
        if not np.isnan(x[0]):
            continue
        out = o.sr_fill(x, 0, 1, 0, rbits=r_all)
        assert np.all(bf16_is_nan(out)), f"NaN {u:#x} did not stay NaN"
        assert np.all((out >> 15) == (u >> 31)), f"NaN {u:#x} lost its sign"
        assert np.all(out == out[0]), f"NaN {u:#x} result depends on the random bits"
        assert np.all(out & 0x0040), f"NaN {u:#x} not quiet"
        rn = o.rne_bf16(x[0])
        assert bf16_is_nan(np.array([rn]))[0], f"RNE of NaN {u:#x} is not NaN"


def pin_sr_mean_with_philox(o):
    """Outputs drawn with the Philox stream average to x (within 5 sigma) and
    land only on the two bracketing values."""
    n = 1 << 16
    for xv, step, seed in ((1.0 + 1e-4, 1, 0), (0.3, 7, 1234), (-2.71828, 3, 2**40 + 5),
                           (1e-30, 2, 9)):
        x = np.full(n, xv, dtype=np.float32)
        out = o.sr_fill(x, 12345, step, seed)
        u = int(bits_from_f32(x[:1])[0])
        lo, p = u >> 16, (u & 0xFFFF) / 65536.0
        assert np.all((out == lo) | (out == lo + 1))
        spacing = abs(bf16_value([lo + 1])[0] - bf16_value([lo])[0])
        sigma = spacing * np.sqrt(max(p * (1 - p), 1e-12) / n)
        mean = bf16_value(out).mean()
        assert abs(mean - float(x[0])) < 5 * sigma + 1e-300, f"x={xv}: mean {mean} vs {x[0]}"


def pin_rne_matches_torch(o, seed=3):
    """Round-to-nearest-even equals torch's float32 -> bfloat16 conversion,
    including exact ties and overflow to Inf."""
    rng = np.random.default_rng(seed)
    pats = rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 2**16, 2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    pats = np.concatenate([pats, ties, sr_edge_patterns(),
                           np.array([0x7F7FFFFF, 0xFF7FFFFF, 0x7F7F8000, 0x7F7F7FFF], np.uint32)])
    pats = pats[~np.isnan(f32_from_bits(pats))]
    x = f32_from_bits(pats)
    want = W.to_bf16_bits(x)
    got = o.rne_fill(x)
    got1 = np.array([o.rne_bf16(v) for v in x[:200]], dtype=np.uint16)
    assert np.array_equal(got[:200], got1)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"RNE differs from torch for {bad.size} inputs, e.g. {pats[bad[:3]]}"


# --------------------------------------------------------------------------
# AdamW
# --------------------------------------------------------------------------

def textbook_adamw_fp64(p, grads, *, lr, beta1, beta2, eps, weight_decay):
    """AdamW (Loshchilov and Hutter) in binary64: bias-corrected moments and
    the decoupled decay term lr*wd*theta."""
    p = p.astype(np.float64).copy()
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    for t, g in enumerate(grads, start=1):
        g = g.astype(np.float64)
        m = beta1 * m + (1 - beta1) * g
        v = beta2 * v + (1 - beta2) * g * g
        mhat = m / (1 - beta1 ** t)
        vhat = v / (1 - beta2 ** t)
        p = p - lr * (mhat / (np.sqrt(vhat) + eps) + weight_decay * p)
    return p


def _fp32_run(o, p0, grads, **hp):
    p = p0.copy()
    m = np.zeros_like(p)
    v = np.zeros_like(p)
    for t, g in enumerate(grads, start=1):
        o.adamw_step(p, g, m, v, step=t, seed=0, **hp)
    return p


def _config2_inputs(n=1 << 16, steps=100, seed=0):
    p0 = W.normal_f32(W.host_rng(seed, 0), n, 0.02)
    grads = [W.normal_f32(W.host_rng(seed, t), n, 1e-3) for t in range(1, steps + 1)]
    return p0, grads


def load_criterion():
    with open(os.path.join(GOLDEN, "adamw_criterion.json")) as f:
        return json.load(f)


def pin_adamw_textbook(o):
    """fp32 oracle vs the binary64 textbook recurrence over 100 steps: within
    the page's 1e-4, and within 2e-6 (fp32 rounding alone is ~1e-7 here)."""
    crit = load_criterion()
    p0, grads = _config2_inputs(steps=crit["steps"])
    got = _fp32_run(o, p0, grads, **HP)
    want = textbook_adamw_fp64(p0, grads, **HP)
    d = np.abs(got.astype(np.float64) - want).max()
    assert d < crit["max_abs_diff"], f"max |diff| {d:.3e} breaks the page's criterion"
    assert d < 2e-6, f"max |diff| {d:.3e} is far above fp32 rounding"


def pin_adamw_torch(o):
    """fp32 oracle vs torch.optim.AdamW (single-tensor path, CPU, fp32) over
    100 steps."""
    import torch
    crit = load_criterion()
    p0, grads = _config2_inputs(n=1 << 15, steps=crit["steps"], seed=1)
    got = _fp32_run(o, p0, grads, **HP)
    tp = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.AdamW([tp], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]),
                            eps=HP["eps"], weight_decay=HP["weight_decay"],
                            foreach=False, fused=False)
    for g in grads:
        tp.grad = torch.from_numpy(g.copy())
        opt.step()
    d = np.abs(got.astype(np.float64) - tp.detach().numpy().astype(np.float64)).max()
    assert d < crit["max_abs_diff"] and d < 2e-6, f"max |diff| vs torch AdamW {d:.3e}"


def pin_adamw_special_cases(o):
    """Closed forms: (a) zero gradient from zero state is pure decay
    p*(1-lr*wd), moments stay 0; (b) from p = 0 the first step is
    -lr*g/(|g|+eps); (c) the same with |g| far below eps (eps-dominated)."""
    rng = np.random.default_rng(4)
    n = 4096
    # (a)
    p = W.normal_f32(rng, n, 0.5)
    p64 = p.astype(np.float64)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    for t in (1, 2, 50):
        o.adamw_step(p, np.zeros(n, np.float32), m, v, step=t, seed=0, **HP)
        p64 = p64 * (1 - HP["lr"] * HP["weight_decay"])
        ulp = np.spacing(np.abs(p).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(p - p64) <= 2 * t * ulp), "zero-gradient step is not the decay"
        assert not m.any() and not v.any(), "moments moved without a gradient"
    # (b) and (c)
    for scale, eps in ((1e-3, 1e-8), (1e-12, 1e-8), (3.0, 1e-3)):
        g = W.normal_f32(rng, n, scale)
        p = np.zeros(n, np.float32)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        hp = dict(HP, eps=eps)
        o.adamw_step(p, g, m, v, step=1, seed=0, **hp)
        g64 = g.astype(np.float64)
        want = -hp["lr"] * g64 / (np.abs(g64) + eps)
        rel = np.abs(p - want) / np.maximum(np.abs(want), 1e-30)
        assert rel.max() < 1e-5, f"first step (|g|~{scale}, eps {eps}) off by {rel.max():.2e}"
        assert np.allclose(m, (1 - HP["beta1"]) * g64, rtol=1e-6, atol=0)
        assert np.allclose(v, (1 - HP["beta2"]) * g64 * g64, rtol=1e-6, atol=0)


def pin_adamw_one_step_tight(o):
    """From a random mid-training state, one fp32 step is within a few fp32
    rounding errors of the same step in binary64."""
    rng = np.random.default_rng(6)
    n = 1 << 15
    p = W.normal_f32(rng, n, 0.02)
    g = W.normal_f32(rng, n, 1e-3)
    m = W.normal_f32(rng, n, 1e-4)
    v = (np.abs(W.normal_f32(rng, n, 1e-6)) + np.float32(1e-8)).astype(np.float32)
    t = 37
    P, G, M, V = (a.astype(np.float64) for a in (p, g, m, v))
    hp = HP
    M1 = hp["beta1"] * M + (1 - hp["beta1"]) * G
    V1 = hp["beta2"] * V + (1 - hp["beta2"]) * G * G
    upd = hp["lr"] / (1 - hp["beta1"] ** t) * M1 / (np.sqrt(V1 / (1 - hp["beta2"] ** t)) + hp["eps"])
    P1 = P * (1 - hp["lr"] * hp["weight_decay"]) - upd
    o.adamw_step(p, g, m, v, step=t, seed=0, **hp)
    tol = 4 * np.spacing(np.abs(P1).astype(np.float32)) + 1e-5 * np.abs(upd)
    assert np.all(np.abs(p - P1) <= tol), "parameter off the binary64 step"
    # the two terms of each moment may cancel: bound by their magnitudes
    scale_m = hp["beta1"] * np.abs(M) + (1 - hp["beta1"]) * np.abs(G)
    assert np.all(np.abs(m - M1) <= 1e-6 * scale_m), "first moment off"
    assert np.all(np.abs(v - V1) <= 1e-6 * V1), "second moment off"


def pin_adamw_dtype_paths(o):
    """A bf16 gradient acts as its exact float32 widening; a bf16 parameter
    with RNE write-back is the fp32-path result rounded by torch's RNE; with
    SR write-back it is that result rounded stochastically with the element's
    own Philox word."""
    rng = np.random.default_rng(8)
    n = 3000
    pb = W.to_bf16_bits(W.normal_f32(rng, n, 0.02))
    gb = W.to_bf16_bits(W.normal_f32(rng, n, 1e-3))
    m0 = W.normal_f32(rng, n, 1e-4)
    v0 = np.abs(W.normal_f32(rng, n, 1e-6))
    pf = W.bf16_bits_to_f32(pb)
    gf = W.bf16_bits_to_f32(gb)
    kw = dict(step=5, seed=99, base_index=1001, **HP)
    # fp32 reference path
    p_ref, m_ref, v_ref = pf.copy(), m0.copy(), v0.copy()
    o.adamw_step(p_ref, gf, m_ref, v_ref, **kw)
    # bf16 grad, f32 param
    p1, m1, v1 = pf.copy(), m0.copy(), v0.copy()
    o.adamw_step(p1, gb, m1, v1, **kw)
    assert np.array_equal(bits_from_f32(p1), bits_from_f32(p_ref))
    assert np.array_equal(bits_from_f32(m1), bits_from_f32(m_ref))
    assert np.array_equal(bits_from_f32(v1), bits_from_f32(v_ref))
    # bf16 param, RNE
    p2, m2, v2 = pb.copy(), m0.copy(), v0.copy()
    o.adamw_step(p2, gb, m2, v2, rounding=1, **kw)
    assert np.array_equal(p2, W.to_bf16_bits(p_ref)), "RNE write-back differs"
    assert np.array_equal(bits_from_f32(m2), bits_from_f32(m_ref))
    # bf16 param, SR
    p3, m3, v3 = pb.copy(), m0.copy(), v0.copy()
    o.adamw_step(p3, gf, m3, v3, rounding=0, **kw)
    words = np.array([o.element_word(1001 + j, 5, 99) for j in range(n)], dtype=np.uint32)
    assert np.array_equal(p3, o.sr_fill(p_ref, 0, 0, 0, rbits=words)), "SR write-back differs"


def pin_scalars(o):
    """The binary32 per-step scalars are their binary64 definitions rounded
    once (checked to 1 binary32 ulp against numpy binary64)."""
    for lr, b1, b2, eps, wd, t in ((1e-3, 0.9, 0.999, 1e-8, 0.01, 1),
                                   (3e-4, 0.95, 0.98, 1e-6, 0.1, 1000),
                                   (1e-2, 0.0, 0.5, 0.0, 0.0, 7),
                                   (1e-3, 0.9, 0.999, 1e-8, 0.01, 4_000_000_000)):
        got = o.adamw_scalars(lr, b1, b2, eps, wd, t).astype(np.float64)
        want = np.array([b1, b2, eps, 1 - lr * wd, 1 - b1, 1 - b2,
                         lr / (1 - b1 ** t), np.sqrt(1 - b2 ** t)], dtype=np.float64)
        ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(got - want) <= ulp), f"scalars {got} vs {want}"


# --------------------------------------------------------------------------
# sub-ULP demonstration ("adamw-sr", introduction)
# --------------------------------------------------------------------------

def load_demo():
    with open(os.path.join(GOLDEN, "subulp_demo.json")) as f:
        return json.load(f)


def pin_demo_increment(o, n=4096):
    """w <- round(w + 1e-4) from 1.0 for 6,000 steps: round-to-nearest never
    moves; stochastic rounding keeps the mean at 1 + k*1e-4 (unbiased)."""
    d = load_demo()
    inc = np.float32(d["update"])
    # the increment w + inc actually makes on the bf16 grid of [1, 2) after
    # the binary32 addition rounds it
    inc_eff = float(np.float32(np.float32(1.0) + inc)) - 1.0
    spacing = 2.0 ** -7
    p = inc_eff / spacing
    w_rn = np.full(n, W.to_bf16_bits(np.array([d["start"]], np.float32))[0], np.uint16)
    w_sr = w_rn.copy()
    var = 0.0
    for k in range(1, d["steps"] + 1):
        x_rn = (W.bf16_bits_to_f32(w_rn) + inc).astype(np.float32)
        w_rn = o.rne_fill(x_rn)
        xs = (W.bf16_bits_to_f32(w_sr) + inc).astype(np.float32)
        w_sr = o.sr_fill(xs, 0, k, 2024)
        var += spacing * spacing * p * (1 - p)
        if k % 1000 == 0:
            mean_rn = bf16_value(w_rn).mean()
            assert mean_rn == d["rn_final_mean"], f"RN moved to {mean_rn} at step {k}"
            mean_sr = bf16_value(w_sr).mean()
            expect = d["start"] + k * inc_eff
            assert abs(mean_sr - expect) < 5 * np.sqrt(var / n), \
                f"SR mean {mean_sr} vs {expect} at step {k}"


def pin_demo_adamw(o, n=2048):
    """AdamW on loss (w - 1.5)^2 from w = 1.0 (bf16, no fp32 master), lr 1e-4,
    6,000 steps: RNE stays exactly 1.0; the SR mean follows the unrounded
    binary64 AdamW trajectory toward the 1.5 target (it is unbiased); two SR
    runs are bitwise identical."""
    d = load_demo()
    hp = dict(lr=d["update"], beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0)
    checkpoints = range(1000, d["steps"] + 1, 1000)

    # the same optimisation without any rounding, in binary64
    ref = {}
    w64, m64, v64 = d["start"], 0.0, 0.0
    for k in range(1, d["steps"] + 1):
        g = 2.0 * (w64 - d["sr_target"])
        m64 = hp["beta1"] * m64 + (1 - hp["beta1"]) * g
        v64 = hp["beta2"] * v64 + (1 - hp["beta2"]) * g * g
        w64 -= hp["lr"] * (m64 / (1 - hp["beta1"] ** k)) / (
            np.sqrt(v64 / (1 - hp["beta2"] ** k)) + hp["eps"])
        ref[k] = w64

    def run(rounding):
        w = np.full(n, W.to_bf16_bits(np.array([d["start"]], np.float32))[0], np.uint16)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        target = np.float32(d["sr_target"])
        means = {}
        for k in range(1, d["steps"] + 1):
            g = (np.float32(2.0) * (W.bf16_bits_to_f32(w) - target)).astype(np.float32)
            o.adamw_step(w, g, m, v, step=k, seed=7, rounding=rounding, **hp)
            if k in checkpoints:
                means[k] = bf16_value(w).mean()
        return w, m, v, means

    w_rn, _, _, means_rn = run(1)
    assert np.all(bf16_value(w_rn) == d["rn_final_mean"]), "round-to-nearest moved the weight"
    w_sr, m_sr, v_sr, means_sr = run(0)
    prev = d["start"]
    for k in checkpoints:
        assert abs(means_sr[k] - ref[k]) < 0.01, f"step {k}: SR mean {means_sr[k]} vs {ref[k]}"
        assert prev < means_sr[k] < d["sr_target"], f"step {k}: SR mean not moving toward the target"
        prev = means_sr[k]
    w2, m2, v2, _ = run(0)
    assert np.array_equal(w_sr, w2) and np.array_equal(m_sr, m2) and np.array_equal(v_sr, v2)


# --------------------------------------------------------------------------
# shard invariance ("adamw-sr", Method and Correctness)
# --------------------------------------------------------------------------

def pin_shard_invariance(o):
    """Whole vs shards with their base_index, at cuts of every residue mod 4
    and 1-element shards: bitwise equal (AdamW-SR and plain SR)."""
    rng = np.random.default_rng(10)
    n = 10007
    base = 2**33 + 2
    pb = W.to_bf16_bits(W.uniform_f32(rng, n, -1, 1))
    gb = W.to_bf16_bits(W.normal_f32(rng, n, 1e-2))
    m0 = W.normal_f32(rng, n, 1e-3)
    v0 = np.abs(W.normal_f32(rng, n, 1e-4))
    kw = dict(step=7, seed=1234, **HP)
    pw, mw, vw = pb.copy(), m0.copy(), v0.copy()
    o.adamw_step(pw, gb, mw, vw, base_index=base, **kw)
    cuts = [0, 1, 2, 3, 5, 6, 7, 8, 1001, 1002, 1003, 4096, 4097, 9999, n]
    ps, ms, vs = pb.copy(), m0.copy(), v0.copy()
    for a, b in zip(cuts[:-1], cuts[1:]):
        sp, sm, sv = ps[a:b].copy(), ms[a:b].copy(), vs[a:b].copy()
        o.adamw_step(sp, gb[a:b].copy(), sm, sv, base_index=base + a, **kw)
        ps[a:b], ms[a:b], vs[a:b] = sp, sm, sv
    assert np.array_equal(ps, pw) and np.array_equal(ms, mw) and np.array_equal(vs, vw)
    x = W.normal_f32(rng, n, 1.0)
    whole = o.sr_fill(x, base, 3, 5)
    parts = np.concatenate([o.sr_fill(x[a:b], base + a, 3, 5) for a, b in zip(cuts[:-1], cuts[1:])])
    assert np.array_equal(whole, parts)
    # a different seed or step changes the bits
    assert not np.array_equal(whole, o.sr_fill(x, base, 4, 5))
    assert not np.array_equal(whole, o.sr_fill(x, base, 3, 6))


# --------------------------------------------------------------------------
# build flags
# --------------------------------------------------------------------------

def pin_no_contraction(o):
    """The oracle build rounds a*b and (a*b)+c separately (no FMA): with
    a = b = 1+2^-12 and c = -(1+2^-11) the unfused result is 0, the fused 2^-24."""
    a = float(np.float32(1 + 2**-12))
    c = float(np.float32(-(1 + 2**-11)))
    assert o.mul_add(a, a, c) == 0.0


# --------------------------------------------------------------------------
# bf16 GEMM with a stochastic-rounding epilogue ("Add stochastic rounding and
# philox RNG helpers", Consumer)
# --------------------------------------------------------------------------

def _bf16_grid(rng, shape, emin=-6, emax=6):
    """bf16 patterns of values m * 2^e, |m| < 256 an integer, e in [emin, emax]:
    sums of a few such products are exact in binary64."""
    mant = rng.integers(-255, 256, size=shape).astype(np.float64)
    expo = rng.integers(emin, emax + 1, size=shape).astype(np.float64)
    return W.to_bf16_bits((mant * 2.0 ** (expo - 7)).astype(np.float32))


def pin_gemm_exact_small(o, seed=5):
    """C = A.B^T on 3 x 7 by 5 x 7 operands (non-square: a transposed operand
    or a swapped index cannot pass): the accumulator equals the exact rational
    sum rounded once to binary32; element (row0+i, j) is rounded with word
    (row0+i)*n + j of the Philox stream (or to nearest-even); computing the
    rows from row0 in two slices gives the same bits as the whole."""
    from fractions import Fraction
    rng = np.random.default_rng(seed)
    m, n, k = 3, 5, 7
    a = _bf16_grid(rng, (m, k))
    b = _bf16_grid(rng, (n, k))
    av, bv = bf16_value(a), bf16_value(b)
    exact = np.zeros((m, n), dtype=np.float32)
    for i in range(m):
        for j in range(n):
            s = sum((Fraction(float(av[i, t])) * Fraction(float(bv[j, t])) for t in range(k)), Fraction(0))
            exact[i, j] = np.float32(float(s))          # float(s) is exact here; one rounding to binary32
    row0, step, seed_ = 1000, 9, 2**37 + 5
    out, acc = o.gemm_bf16(a, b, row0=row0, step=step, seed=seed_)
    assert np.array_equal(bits_from_f32(acc), bits_from_f32(exact)), "accumulator is not the exact sum"
    for i in range(m):
        for j in range(n):
            r = o.element_word((row0 + i) * n + j, step, seed_)
            assert int(out[i, j]) == o.sr_bf16(exact[i, j], r), f"SR element ({i}, {j})"
    out_rn, _ = o.gemm_bf16(a, b, row0=row0, rounding=1)
    assert np.array_equal(out_rn, o.rne_fill(exact)), "RNE epilogue"
    top, _ = o.gemm_bf16(a[:1], b, row0=row0, step=step, seed=seed_)
    rest, _ = o.gemm_bf16(a[1:], b, row0=row0 + 1, step=step, seed=seed_)
    assert np.array_equal(np.vstack([top, rest]), out), "row slices differ from the whole"


def pin_gemm_closed_forms(o, seed=6):
    """Products that are exactly bf16 values come out unchanged for every
    seed and both roundings: (a) one-hot rows of A pick C[i, j] = B[j, sel_i];
    (b) entries in {-2..2} with k = 24 give integer sums |s| <= 96."""
    rng = np.random.default_rng(seed)
    m, n, k = 6, 10, 12
    sel = rng.integers(0, k, size=m)
    a = np.zeros((m, k), dtype=np.uint16)
    a[np.arange(m), sel] = 0x3F80                                   # 1.0
    b = W.to_bf16_bits(rng.normal(0.0, 3.0, size=(n, k)).astype(np.float32))
    want = b[:, sel].T.copy()
    for s_ in (0, 1, 2**63 + 11):
        out, _ = o.gemm_bf16(a, b, row0=17, step=3, seed=s_)
        assert np.array_equal(out, want), f"one-hot rows, seed {s_}"
    out, _ = o.gemm_bf16(a, b, rounding=1)
    assert np.array_equal(out, want), "one-hot rows, RNE"
    ai = rng.integers(-2, 3, size=(7, 24)).astype(np.float32)
    bi = rng.integers(-2, 3, size=(9, 24)).astype(np.float32)
    want = W.to_bf16_bits((ai @ bi.T).astype(np.float32))
    for s_ in (4, 5):
        out, _ = o.gemm_bf16(W.to_bf16_bits(ai), W.to_bf16_bits(bi), step=1, seed=s_)
        assert np.array_equal(out, want), f"integer sums, seed {s_}"
