"""Peaked score distributions: one dominant token per (sequence, KV head) segment.

"From MHA to MLA", section 2: the weights P are rounded to the value dtype before the
PV product (``p.to(V.dtype)``). When one token carries most of the softmax mass, the
rounding error of that one weight goes straight into the output, so these cases check
every decode kernel in the regime where the rounding of P matters most.

Construction (host only, numpy; no attention arithmetic of the oracle is reused):
  * a "marker" block of dims (GQA: the last 16 dims of each head; MLA: the 64 rope
    dims) is set to 1 in every query row and to 0 in every cached key, so it adds
    nothing to an ordinary token's score;
  * the dominant token t* gets marker value c and a content part that every query row
    of its segment is orthogonal to, so its score is scale * width * c for every row;
    its value row reaches the clip bound vmax of all values (vmax = 2 keeps the bf16
    rounding of the output at most 2^-8; vmax = 3.9 leaves a kernel that normalises by
    the sum of the unrounded weights no margin);
  * decoys sit a little below the dominant score (GQA: one token a page earlier, 5
    below; MLA: slot 0 of every page, 5.3 below), so a kernel whose running maximum is
    raised only by large jumps keeps a decoy's maximum and weighs t* by a
    non-power-of-two factor that rounding changes;
  * c is chosen from the realized scores of the other tokens so that t* carries the
    requested share of its row's softmax mass (averaged over the segment's rows).
"""
from __future__ import annotations

import numpy as np

from paged_kv_cache_61_gb300 import synth


def _f32(bits, dtype):
    return synth.bits_to_float32(np.asarray(bits), dtype).astype(np.float64)


def _bits(x, dtype):
    return synth.float32_to_bits(np.asarray(x, dtype=np.float32), dtype)


def _token_slot(case, b, t):
    p = case.page_size
    return int(case.block_tables[b, t // p]), t % p


def _orthogonal_value(rng, q_rows, width, vmax):
    """A vector of ``width`` entries, |entry| in [0.75 vmax, vmax] before the projection,
    orthogonal to every row of q_rows (projected onto their null space), rescaled so the
    largest entry is vmax."""
    x = rng.choice([-1.0, 1.0], size=width) * rng.uniform(0.75 * vmax, vmax, size=width)
    if q_rows.shape[0]:
        u, s, vt = np.linalg.svd(q_rows, full_matrices=True)
        rank = int((s > 1e-9 * s.max()).sum())
        basis = vt[rank:]                       # null space of q_rows
        x = basis.T @ (basis @ x)
    return x * (vmax / np.abs(x).max())


def _marker_value(z_rest, weight, scale, width):
    """Marker value c with exp(scale*width*c) / (exp(...) + Z) = weight for the mean Z."""
    z = float(np.mean(z_rest))
    return float(np.log(weight / (1.0 - weight) * z) / (scale * width))


def plant_gqa(case, weights, seed=0, vmax=2.0):
    """One dominant token per (sequence, KV head) of a GQA case (S = 1), in place.

    weights[b]: the share of the softmax mass of the dominant token of sequence b.
    vmax: every value is clipped to [-vmax, vmax]; the dominant value row reaches it.
    Returns [(b, kvh, t*)].
    """
    rng = np.random.default_rng(seed)
    dt, D, G = case.dtype, case.head_dim_qk, case.group
    W = 16
    q = _f32(case.q, dt)
    k = _f32(case.k_cache, dt)
    v = np.clip(_f32(case.v_cache, dt), -vmax, vmax)
    q[..., D - W:] = 1.0
    k[..., D - W:] = 0.0
    placed = []
    for b, ctx in enumerate(case.context_lens):
        ctx = int(ctx)
        for kvh in range(case.num_kv_heads):
            rows = q[b, kvh * G:(kvh + 1) * G]                    # [G, D]
            ts = int(rng.integers(min(ctx - 1, case.page_size), ctx))
            td = ts - case.page_size if ts >= case.page_size else None
            pb, ps = _token_slot(case, b, ts)
            k[pb, ps, kvh, :] = 0.0
            v[pb, ps, kvh, :] = _orthogonal_value(rng, np.zeros((0, D)), D, vmax)
            if td is not None:
                db, dsl = _token_slot(case, b, td)
                k[db, dsl, kvh, :] = 0.0
            others = [t for t in range(ctx) if t != ts and t != td]
            z = np.zeros(G)
            if others:
                loc = [_token_slot(case, b, t) for t in others]
                keys = np.stack([k[pb2, ps2, kvh] for pb2, ps2 in loc])
                z = np.exp(case.scale * rows @ keys.T).sum(axis=1)
            c = _marker_value(np.maximum(z, 1e-30), weights[b], case.scale, W)
            k[pb, ps, kvh, D - W:] = c
            if td is not None:
                k[db, dsl, kvh, D - W:] = c - 5.0 / (case.scale * W)
            placed.append((b, kvh, ts))
    case.q = _bits(q, dt)
    case.k_cache = _bits(k, dt)
    case.v_cache = _bits(v, dt)
    return placed


def plant_mla(case, weights, seed=0, vmax=2.0):
    """One dominant token per sequence of an MLA case (S = 1), in place.

    Its latent (the value) is orthogonal to the content part of every query head of the
    sequence, so its score is the rope part alone. Slot 0 of every page holds a decoy
    scoring 5.3 below it (7.65 in log2 units): whatever page a piece starts on, its first
    page's maximum is then within 2^8 of the dominant score, so a running maximum that is
    raised only by larger jumps stays below it and the dominant token's weight is a
    non-power-of-two factor that rounding changes. Returns [(b, t*)].
    """
    rng = np.random.default_rng(seed)
    dt, Dv, Dqk, P = case.dtype, case.head_dim_v, case.head_dim_qk, case.page_size
    W = Dqk - Dv
    gap = 5.3
    q = _f32(case.q, dt)
    kv = _f32(case.kv_cache, dt)
    kv[..., :Dv] = np.clip(kv[..., :Dv], -vmax, vmax)
    q[..., Dv:] = 1.0
    kv[..., Dv:] = 0.0
    placed = []
    qr = _f32(_bits(q, dt), dt)                  # the rows the kernels will see
    for b, ctx in enumerate(case.context_lens):
        ctx = int(ctx)
        cand = [t for t in range(ctx) if t % P != 0]
        ts = int(cand[int(rng.integers(len(cand) // 2, len(cand)))])
        decoys = list(range(0, ctx, P))
        pb, ps = _token_slot(case, b, ts)
        kv[pb, ps, :] = 0.0
        kv[pb, ps, :Dv] = _orthogonal_value(rng, qr[b, :, :Dv], Dv, vmax)
        for t in decoys:                 # latent 0: the decoy's score is its rope part
            db, dsl = _token_slot(case, b, t)
            kv[db, dsl, :] = 0.0
        others = [t for t in range(ctx) if t != ts and t % P != 0]
        loc = [_token_slot(case, b, t) for t in others]
        rec = np.stack([kv[pb2, ps2] for pb2, ps2 in loc])
        z = np.exp(case.scale * qr[b] @ rec.T).sum(axis=1)          # ordinary tokens
        # exp(s*) (1 - w (1 + n_d e^-gap)) = w Z
        w = weights[b]
        frac = 1.0 - w * (1.0 + len(decoys) * np.exp(-gap))
        assert frac > 0, "too many decoys for this weight"
        c = float(np.log(w * float(np.mean(z)) / frac) / (case.scale * W))
        kv[pb, ps, Dv:] = c
        for t in decoys:
            db, dsl = _token_slot(case, b, t)
            kv[db, dsl, Dv:] = c - gap / (case.scale * W)
        placed.append((b, ts))
    case.q = _bits(q, dt)
    case.kv_cache = _bits(kv, dt)
    return placed


def dominant_weights_gqa(case, placed):
    """Realized softmax share of each placed token, per query head: {(b, h): w}."""
    dt, G, p = case.dtype, case.group, case.page_size
    q, k = _f32(case.q, dt), _f32(case.k_cache, dt)
    got = {}
    for b, kvh, ts in placed:
        ctx = int(case.context_lens[b])
        loc = [_token_slot(case, b, t) for t in range(ctx)]
        keys = np.stack([k[pb, ps, kvh] for pb, ps in loc])
        for h in range(kvh * G, (kvh + 1) * G):
            s = case.scale * keys @ q[b, h]
            e = np.exp(s - s.max())
            got[(b, h)] = float(e[ts] / e.sum())
    return got


def dominant_weights_mla(case, placed):
    dt = case.dtype
    q, kv = _f32(case.q, dt), _f32(case.kv_cache, dt)
    got = {}
    for b, ts in placed:
        ctx = int(case.context_lens[b])
        rec = np.stack([kv[_token_slot(case, b, t)] for t in range(ctx)])
        s = case.scale * rec @ q[b].T                    # [ctx, Hq]
        e = np.exp(s - s.max(axis=0))
        for h in range(case.num_q_heads):
            got[(b, h)] = float(e[ts, h] / e[:, h].sum())
    return got
