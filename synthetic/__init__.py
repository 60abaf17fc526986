"""Seeded synthetic inputs for the drafter-sampling hot path.

This module only *makes inputs*: random tables, logits, hidden states,
weights, token-id streams and the explicit uniforms that the method consumes.
It holds none of the method's arithmetic (no softmax over a vocabulary that
the method computes, no acceptance test, no residual, no inverse-CDF draw with
the method's uniforms).  Both the CPU oracle and the CUDA library receive the
arrays made here; neither imports the other.

Every generator is a numpy ``Generator`` over the Philox counter-based bit
generator (Salmon et al., SC'11), seeded explicitly, so a workload is a pure
function of its seed.  The workload recipes follow the five configurations of
the drafter-sampling study:

* toy   : V=18, 19 contexts, Dirichlet(1) target rows, q_w = w p + (1-w) q0
* head  : hidden [B,2048] bf16 N(0,1), W [128256,2048] bf16 N(0,0.02),
          top-K (K=32768) of a Zipf(1.1) frequency table
* verify: B=16, gamma=6, V=128256, K=32768, fp32 logits
          N(0,2) + 3 ln Zipf_1.1(rank), q = softmax over the trimmed ids of
          (logit + N(0,1)), drafted tokens sampled from q
* calib : 50M ids Zipf(1.1) over V=128256, W [128256,3072] bf16 N(0,0.02)
* large : B=256, gamma=8, V=152064, H=4096, K=38016 (Zipf 1.05 ranking),
          bf16 logits built like ``verify``, T=0.7

"N(mu, s)" is read with s the standard deviation.  The rank -> token-id map
is a seeded permutation, so frequent ids are scattered over [0, V) as in a
real tokenizer.
"""
from __future__ import annotations

import numpy as np

# Seeds fixed by the workload recipes.
SEED_TOY = 0
SEED_VERIFY = 1
SEED_CALIB = 2
SEED_PERM = 7


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """Philox-backed generator; ``stream`` selects an independent key."""
    return np.random.Generator(np.random.Philox(key=[int(seed), int(stream)]))


def uniforms(seed: int, stream: int, shape) -> np.ndarray:
    """float32 uniforms in [0, 1) (24-bit resolution)."""
    return rng(seed, stream).random(shape, dtype=np.float32)


# --------------------------------------------------------------------- bf16
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Quantise float32 values to bfloat16 (round to nearest even).

    Returns the raw 16-bit patterns as uint16.  Inputs are finite.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(g: np.random.Generator, shape, std: float,
                chunk: int = 1 << 24) -> np.ndarray:
    """N(0, std) samples quantised to bf16 bit patterns, generated in chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = g.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s:e] = to_bf16_bits(v)
    return out.reshape(shape)


# --------------------------------------------------------------- Zipf tables
def zipf_pmf(V: int, s: float) -> np.ndarray:
    """pmf over ranks 1..V proportional to r^-s (float64)."""
    r = np.arange(1, V + 1, dtype=np.float64)
    w = r ** (-float(s))
    return w / w.sum()


def rank_permutation(V: int, seed: int = SEED_PERM) -> np.ndarray:
    """perm[r] = token id of rank r (0-based rank)."""
    return rng(seed, 99).permutation(V).astype(np.int32)


def trimmed_set(V: int, K: int, perm: np.ndarray):
    """The K most frequent ids of a Zipf table (ranks 0..K-1 under ``perm``).

    Returns (ranked_ids, trim_ids ascending, inv_map with -1 for absent ids).
    Used to give verify and draft workloads the trimmed vocabulary that a
    calibration on the frequency table (not a sampled stream) would produce.
    """
    ranked = perm[:K].astype(np.int32)
    trim_ids = np.sort(ranked).astype(np.int32)
    inv_map = np.full(V, -1, dtype=np.int32)
    inv_map[trim_ids] = np.arange(K, dtype=np.int32)
    return ranked, trim_ids, inv_map


def rank_bias(V: int, s: float, perm: np.ndarray, scale: float = 3.0) -> np.ndarray:
    """bias[id] = scale * ln pmf(rank(id)) for a Zipf(s) table (float64)."""
    lp = np.log(zipf_pmf(V, s))
    bias = np.empty(V, dtype=np.float64)
    bias[perm] = scale * lp
    return bias


# ------------------------------------------------------------- toy workload
def toy_tables(V: int = 18, w: float = 0.5, seed: int = SEED_TOY):
    """Dirichlet(1) target rows for BOS + V contexts, a Dirichlet(1) unigram
    q0, and the mixture draft q_w = w p + (1-w) q0.

    Context index 0 is BOS; context c = t + 1 follows token t.
    Returns float64 arrays p [V+1, V], q0 [V], q_w [V+1, V].
    """
    g = rng(seed, 0)
    p = g.dirichlet(np.ones(V), size=V + 1)
    q0 = g.dirichlet(np.ones(V))
    q_w = w * p + (1.0 - w) * q0[None, :]
    return p, q0, q_w


def toy_drafts(g: np.random.Generator, q_w: np.ndarray, ctx: int, gamma: int) -> np.ndarray:
    """Draft gamma tokens from the toy mixture draft, each conditioned on the
    previous token (the toy drafter stands in for a draft model)."""
    V = q_w.shape[1]
    out = np.empty(gamma, dtype=np.int32)
    c = ctx
    for i in range(gamma):
        out[i] = g.choice(V, p=q_w[c])
        c = int(out[i]) + 1
    return out


# ----------------------------------------------------------- verify workload
def softmax_rows_for_inputs(x: np.ndarray) -> np.ndarray:
    """Plain row softmax used only to *build* synthetic draft distributions."""
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def verify_inputs(B: int = 16, gamma: int = 6, V: int = 128256, K: int = 32768,
                  seed: int = SEED_VERIFY, s_target: float = 1.1,
                  logits_dtype: str = "f32", noise_std: float = 1.0,
                  identity_perm: bool = False):
    """Batched-verify workload.

    logits[b,i,:] = N(0,2) + 3 ln Zipf_{s_target}(rank)   (float32, or bf16 bits)
    q[b,i,:]      = softmax over the trimmed ids of (logit + N(0, noise_std))
    draft[b,i]    ~ q[b,i]  (target ids), sampled by numpy's Generator
    u_accept [B,gamma], u_resample [B,gamma+1]: Philox uniforms.

    The trimmed set is the top-K ranks under the rank permutation.  Any Zipf
    exponent ranks ids in the same order, so the large-batch recipe's
    "s=1.05 ranking" selects the same top-K ranks.
    """
    perm = np.arange(V, dtype=np.int32) if identity_perm else rank_permutation(V)
    ranked, trim_ids, inv_map = trimmed_set(V, K, perm)
    bias = rank_bias(V, s_target, perm).astype(np.float32)

    R = gamma + 1
    g = rng(seed, 1)
    gq = rng(seed, 2)
    gd = rng(seed, 3)
    if logits_dtype == "bf16":
        logits = np.empty((B, R, V), dtype=np.uint16)
    else:
        logits = np.empty((B, R, V), dtype=np.float32)
    q32 = np.empty((B, gamma, K), dtype=np.float32)
    draft = np.empty((B, gamma), dtype=np.int32)
    for b in range(B):
        lb = g.standard_normal((R, V), dtype=np.float32) * np.float32(2.0) + bias[None, :]
        if logits_dtype == "bf16":
            logits[b] = to_bf16_bits(lb)
            l_for_q = (logits[b].astype(np.uint32) << np.uint32(16)).view(np.float32)
        else:
            logits[b] = lb
            l_for_q = lb
        x = l_for_q[:gamma][:, trim_ids].astype(np.float64)
        x += gq.standard_normal((gamma, K)) * noise_std
        q32[b] = softmax_rows_for_inputs(x).astype(np.float32)
        for i in range(gamma):
            pr = q32[b, i].astype(np.float64)
            pr /= pr.sum()
            draft[b, i] = trim_ids[gd.choice(K, p=pr)]

    u_acc = uniforms(seed, 4, (B, gamma))
    u_res = uniforms(seed, 5, (B, R))
    return dict(logits=logits, logits_dtype=logits_dtype, q=q32, trim_ids=trim_ids,
                inv_map=inv_map, ranked_ids=ranked, draft=draft, u_accept=u_acc,
                u_resample=u_res, B=B, gamma=gamma, V=V, K=K)


# ------------------------------------------------------------- head workload
def head_weights(V: int, H: int, seed: int, std: float = 0.02) -> np.ndarray:
    """LM-head weights W [V, H], bf16 bits, N(0, std)."""
    return normal_bf16(rng(seed, 10), (V, H), std)


def hidden_states(shape, seed: int, stream: int = 11) -> np.ndarray:
    """Drafter hidden states, bf16 bits, N(0,1)."""
    return normal_bf16(rng(seed, stream), shape, 1.0)


def gather_rows(W: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Plain row selection used to give draft workloads a ready W_trim."""
    return np.ascontiguousarray(W[ids])


# ------------------------------------------------------------ calib workload
def zipf_ids(N: int, V: int, s: float = 1.1, seed: int = SEED_CALIB,
             perm: np.ndarray | None = None, chunk: int = 1 << 23) -> np.ndarray:
    """N token ids: ranks drawn from Zipf(s) over V ranks by inverse-CDF of the
    pmf on uniforms, mapped to ids by the rank permutation.  int32."""
    if perm is None:
        perm = rank_permutation(V)
    cdf = np.cumsum(zipf_pmf(V, s))
    g = rng(seed, 20)
    out = np.empty(N, dtype=np.int32)
    for st in range(0, N, chunk):
        e = min(N, st + chunk)
        u = g.random(e - st)
        r = np.searchsorted(cdf, u, side="right")
        np.minimum(r, V - 1, out=r)
        out[st:e] = perm[r]
    return out
