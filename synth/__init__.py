"""Seeded synthetic inputs for verification and OPD-loss workloads.

This module only makes inputs: logits with the stated distributions, ragged
lengths packed by CSR offsets, and draft tokens drawn from the draft's own
temperature softmax.  It holds none of the verification or loss arithmetic and
is the one module that both the CUDA path's tests/benchmark and the oracle
consume.  Every array is a pure function of the data seed.

Logits are produced in float32 and rounded to bf16 (round to nearest even);
bf16 tensors are carried as uint16 bit patterns so that the oracle and the GPU
read identical bits.

Draft tokens are drawn with the Gumbel-max rule (x = argmax_v z_v/T + G_v with
G_v standard Gumbel, in float64), which samples exactly from softmax(z/T); at
T = 0 the drafter is greedy (argmax z, smallest index).

Workload presets (the five verification / OPD workloads this library is
measured on):
  1  tiny       N=4, L=16 (+bonus), V=1024, fp32; y~N(0,2^2); z=y+N(0,1); T=1
  2  fixed      N=32, L=16, V=151936, bf16; y~N(0,3^2); z=y+N(0,s_i^2),
                s_i~U[0.5,3] per request; T=1
  3  ragged     N=128, L_i~U{2,4,8,16}, V=151936, bf16; y~N(0,3^2);
                z_j=y_j+N(0,s_j^2), s_j=0.5+2.5 j/15 by position; T=1
  4  opd        64x16 draft rows paired 1:1 with target rows, V=151936, bf16;
                y~N(0,3^2), z=0.7y+N(0,2^2); T=1, c=1, lambda=0.1
  5  mix        N=256, L_i~U{2,4,8,16}, V=151936, bf16; y_v=-1.1 ln rank_pi(v)
                + N(0,1) with pi a per-request random permutation of the vocab;
                z as in preset 3; verify at T in {0, 0.6, 1}, then OPD (T=1)
                on the same batch
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

V_WIDE = 151936
BLOCK_ROWS = 32  # rows per independently seeded generator block

_THREADS = max(1, min(16, os.cpu_count() or 1))


# ---------------------------------------------------------------------------
# bf16 bit patterns
# ---------------------------------------------------------------------------
def bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    nan = np.isnan(x)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def as_f32(a) -> np.ndarray:
    """Logits as float32 values (exact for both bf16 bits and fp32)."""
    a = np.asarray(a)
    return bf16_to_f32(a) if a.dtype == np.uint16 else a.astype(np.float32, copy=False)


# ---------------------------------------------------------------------------
# batch container
# ---------------------------------------------------------------------------
@dataclass
class Batch:
    name: str
    V: int
    dtype: str                 # "bf16" or "f32"
    cu: np.ndarray             # int32 [N+1] CSR offsets of draft rows
    target: np.ndarray         # [rows_t, V] uint16 (bf16 bits) or float32
    draft: np.ndarray          # [rows_d, V]
    tokens: dict = field(default_factory=dict)   # temperature -> int32 [rows_d]
    has_bonus: bool = True     # target rows follow the verify layout
    temperatures: tuple = (1.0,)
    seed: int = 0              # Philox verification seed
    opd: dict = field(default_factory=dict)      # OPD parameters, if any

    @property
    def N(self) -> int:
        return int(self.cu.shape[0] - 1)

    @property
    def total_rows(self) -> int:
        return int(self.cu[-1])

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.cu)

    def esize(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def request_rows(self, i: int):
        """(target row range, draft row range) of request i in the verify layout."""
        c0, c1 = int(self.cu[i]), int(self.cu[i + 1])
        return (c0 + i, c1 + i + 1), (c0, c1)

    def subset(self, reqs):
        """Compact copy holding only requests `reqs` (rows re-packed)."""
        reqs = [int(r) for r in reqs]
        t_rows, d_rows, lens = [], [], []
        for i in reqs:
            (t0, t1), (d0, d1) = self.request_rows(i)
            t_rows.append(np.arange(t0, t1))
            d_rows.append(np.arange(d0, d1))
            lens.append(d1 - d0)
        ti = np.concatenate(t_rows)
        di = np.concatenate(d_rows)
        cu = np.zeros(len(reqs) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        return Batch(name=self.name + "-subset", V=self.V, dtype=self.dtype, cu=cu,
                     target=self.target[ti], draft=self.draft[di],
                     tokens={T: tok[di] for T, tok in self.tokens.items()},
                     has_bonus=self.has_bonus, temperatures=self.temperatures,
                     seed=self.seed, opd=dict(self.opd))


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------
def _block_rngs(seed: int, tag: int, nblocks: int):
    ss = np.random.SeedSequence([seed, tag])
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(nblocks)]


def _parallel_rows(nrows: int, fn):
    """Call fn(block_index, r0, r1) over fixed row blocks (order-independent)."""
    blocks = [(b, r0, min(r0 + BLOCK_ROWS, nrows))
              for b, r0 in enumerate(range(0, nrows, BLOCK_ROWS))]
    if len(blocks) <= 1 or _THREADS == 1:
        for blk in blocks:
            fn(*blk)
        return
    with ThreadPoolExecutor(_THREADS) as ex:
        list(ex.map(lambda blk: fn(*blk), blocks))


def ragged_lengths(rng: np.random.Generator, N: int, choices=(2, 4, 8, 16)) -> np.ndarray:
    return rng.choice(np.asarray(choices, dtype=np.int32), size=N).astype(np.int32)


def cu_from_lengths(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(lengths.shape[0] + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    return cu.astype(np.int32)


def sample_tokens(draft, T: float, seed: int, tag: int = 7) -> np.ndarray:
    """Draft tokens: Gumbel-max draw from softmax(draft/T); argmax at T == 0."""
    z = draft
    R = z.shape[0]
    out = np.zeros(R, dtype=np.int32)
    rngs = _block_rngs(seed, 100 + tag, (R + BLOCK_ROWS - 1) // BLOCK_ROWS)

    def work(b, r0, r1):
        zz = as_f32(z[r0:r1]).astype(np.float64)
        if T == 0.0:
            out[r0:r1] = np.argmax(zz, axis=1)
            return
        u = rngs[b].random(zz.shape)
        # standard Gumbel noise; u == 0 has probability 2^-53 per draw
        g = -np.log(-np.log(np.maximum(u, 1e-300)))
        out[r0:r1] = np.argmax(zz / T + g, axis=1)

    _parallel_rows(R, work)
    return out


def filter_mask(row, T: float, top_k: int, top_p: float) -> np.ndarray:
    """Kept entries of one row under top-k then top-p (order: logit
    descending, smaller index first among equals; top_p is a fraction of the
    top-k set's probability).  Used to draw filtered draft tokens."""
    y = np.asarray(row, dtype=np.float64)
    V = y.shape[0]
    k = top_k if 1 <= top_k < V else V
    if k < V:
        # the k-th largest value, then ties at it in index order
        kth = np.partition(-y, k - 1)[k - 1]
        above = np.nonzero(-y < kth)[0]
        ties = np.nonzero(-y == kth)[0][: k - above.shape[0]]
        cand = np.concatenate([above, ties])
    else:
        cand = np.arange(V)
    cand = cand[np.lexsort((cand, -y[cand]))]
    e = np.exp((y[cand] - y[cand[0]]) / T)
    c = np.cumsum(e)
    n = int(np.searchsorted(c, top_p * c[-1], side="left")) + 1 if top_p < 1.0 else cand.shape[0]
    keep = np.zeros(V, dtype=bool)
    keep[cand[:min(n, cand.shape[0])]] = True
    return keep


def sample_tokens_filtered(draft, T: float, top_k: int, top_p: float, seed: int, tag: int = 9) -> np.ndarray:
    """Draft tokens from the top-k / top-p filtered softmax(draft/T): Gumbel-max
    over the kept entries."""
    z = draft
    R = z.shape[0]
    out = np.zeros(R, dtype=np.int32)
    rngs = _block_rngs(seed, 100 + tag, (R + BLOCK_ROWS - 1) // BLOCK_ROWS)

    def work(b, r0, r1):
        zz = as_f32(z[r0:r1]).astype(np.float64)
        u = rngs[b].random(zz.shape)
        g = -np.log(-np.log(np.maximum(u, 1e-300)))
        for q in range(r1 - r0):
            keep = filter_mask(zz[q], T, top_k, top_p)
            s = np.where(keep, zz[q] / T + g[q], -np.inf)
            out[r0 + q] = int(np.argmax(s))

    _parallel_rows(R, work)
    return out


def make_batch(name: str, *, seed: int, lengths, V: int, dtype: str = "bf16",
               target_kind: str = "normal", target_sd: float = 3.0,
               zipf_s: float = 1.1, draft_kind: str = "add",
               sigma_req=None, sigma_pos=None, draft_scale: float = 0.7,
               draft_sd: float = 2.0, temperatures=(1.0,), has_bonus: bool = True,
               verify_seed: int = 0, opd=None) -> Batch:
    """Build one synthetic batch.

    target_kind: "normal" (y ~ N(0, target_sd^2) iid) or "zipf"
        (y_v = -zipf_s ln rank_pi(v) + N(0, 1), pi per request).
    draft_kind: "add" (z = y + N(0, s^2) with s from sigma_req[i] or
        sigma_pos(j)) or "scaled" (z = draft_scale * y + N(0, draft_sd^2)).
    has_bonus: True -> verify layout (L_i + 1 target rows per request);
        False -> one target row per draft row (OPD pairing 1:1).
    """
    lengths = np.asarray(lengths, dtype=np.int32)
    N = lengths.shape[0]
    cu = cu_from_lengths(lengths)
    R = int(cu[-1])
    rows_t = R + N if has_bonus else R
    # per target row: (request, position j) ; position L_i is the bonus row
    t_req = np.empty(rows_t, dtype=np.int64)
    t_pos = np.empty(rows_t, dtype=np.int64)
    d_trow = np.empty(R, dtype=np.int64)   # target row each draft row pairs with
    for i in range(N):
        L = int(lengths[i])
        n_t = L + 1 if has_bonus else L
        t0 = int(cu[i]) + (i if has_bonus else 0)
        t_req[t0:t0 + n_t] = i
        t_pos[t0:t0 + n_t] = np.arange(n_t)
        d_trow[int(cu[i]):int(cu[i + 1])] = t0 + np.arange(L)

    store = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((rows_t, V), dtype=store)
    draft = np.empty((R, V), dtype=store)
    y32 = np.empty((rows_t, V), dtype=np.float32) if R else None

    base = None
    if target_kind == "zipf":
        rng_p = _block_rngs(seed, 11, 1)[0]
        ranks = np.arange(1, V + 1, dtype=np.float64)
        zipf_base = (-zipf_s * np.log(ranks)).astype(np.float32)
        base = np.empty((N, V), dtype=np.float32)
        for i in range(N):
            base[i, rng_p.permutation(V)] = zipf_base  # token pi^-1(r) gets rank r

    trngs = _block_rngs(seed, 1, (rows_t + BLOCK_ROWS - 1) // BLOCK_ROWS)

    def make_target(b, r0, r1):
        g = trngs[b]
        if target_kind == "normal":
            y = g.standard_normal((r1 - r0, V), dtype=np.float32) * np.float32(target_sd)
        elif target_kind == "zipf":
            y = g.standard_normal((r1 - r0, V), dtype=np.float32)
            y += base[t_req[r0:r1]]
        else:
            raise ValueError(target_kind)
        y32[r0:r1] = y
        target[r0:r1] = bf16_bits(y) if dtype == "bf16" else y

    _parallel_rows(rows_t, make_target)

    drngs = _block_rngs(seed, 2, (R + BLOCK_ROWS - 1) // BLOCK_ROWS)
    d_req = np.repeat(np.arange(N), lengths)
    d_pos = np.concatenate([np.arange(L) for L in lengths]) if N else np.zeros(0, np.int64)

    def make_draft(b, r0, r1):
        g = drngs[b]
        e = g.standard_normal((r1 - r0, V), dtype=np.float32)
        y = y32[d_trow[r0:r1]]
        if draft_kind == "add":
            if sigma_req is not None:
                s = np.asarray(sigma_req, dtype=np.float32)[d_req[r0:r1]]
            else:
                s = np.asarray([sigma_pos(int(j)) for j in d_pos[r0:r1]], dtype=np.float32)
            z = y + e * s[:, None]
        elif draft_kind == "scaled":
            z = np.float32(draft_scale) * y + np.float32(draft_sd) * e
        else:
            raise ValueError(draft_kind)
        draft[r0:r1] = bf16_bits(z) if dtype == "bf16" else z

    _parallel_rows(R, make_draft)
    del y32

    toks = {float(T): sample_tokens(draft, float(T), seed, tag=int(round(T * 1000)))
            for T in temperatures}
    return Batch(name=name, V=V, dtype=dtype, cu=cu, target=target, draft=draft,
                 tokens=toks, has_bonus=has_bonus, temperatures=tuple(temperatures),
                 seed=verify_seed, opd=dict(opd or {}))


def sigma_ramp(j: int) -> float:
    """Draft noise growing linearly along the block: 0.5 at j=0 to 3 at j=15."""
    return 0.5 + 2.5 * min(j, 15) / 15.0


def config(cfg: int, *, N=None, V=None, lengths=None, seed=None) -> Batch:
    """The five workload presets; N / V / lengths may be overridden for
    smaller parity cases of the same shape family."""
    ds = 1000 + cfg if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([ds, 0])))
    if cfg == 1:
        N = N or 4
        lengths = np.full(N, 16, np.int32) if lengths is None else lengths
        return make_batch("tiny", seed=ds, lengths=lengths, V=V or 1024, dtype="f32",
                          target_sd=2.0, sigma_req=np.ones(N), temperatures=(1.0,))
    if cfg == 2:
        N = N or 32
        lengths = np.full(N, 16, np.int32) if lengths is None else lengths
        sig = rng.uniform(0.5, 3.0, size=N)
        return make_batch("fixed", seed=ds, lengths=lengths, V=V or V_WIDE,
                          target_sd=3.0, sigma_req=sig, temperatures=(1.0,))
    if cfg == 3:
        N = N or 128
        lengths = ragged_lengths(rng, N) if lengths is None else lengths
        return make_batch("ragged", seed=ds, lengths=lengths, V=V or V_WIDE,
                          target_sd=3.0, sigma_pos=sigma_ramp, temperatures=(1.0,))
    if cfg == 4:
        N = N or 64
        lengths = np.full(N, 16, np.int32) if lengths is None else lengths
        return make_batch("opd", seed=ds, lengths=lengths, V=V or V_WIDE, target_sd=3.0,
                          draft_kind="scaled", draft_scale=0.7, draft_sd=2.0,
                          temperatures=(), has_bonus=False,
                          opd=dict(temperature=1.0, clip_c=1.0, lambda_ce=0.1))
    if cfg == 5:
        N = N or 256
        lengths = ragged_lengths(rng, N) if lengths is None else lengths
        return make_batch("mix", seed=ds, lengths=lengths, V=V or V_WIDE,
                          target_kind="zipf", zipf_s=1.1, sigma_pos=sigma_ramp,
                          temperatures=(0.0, 0.6, 1.0),
                          opd=dict(temperature=1.0, clip_c=1.0, lambda_ce=0.1))
    raise ValueError(f"unknown preset {cfg}")


def length_head_inputs(N: int, k: int, H: int, Hp: int, seed: int):
    """Synthetic inputs of the adaptive length head: drafter hidden states
    h ~ N(0, 1) (bf16 bits, [N, k, H]) and random weights W1 ~ N(0, 4/H) (bf16
    bits, [H', H]), b1 ~ N(0, 0.3^2), w2 ~ N(0, 4/H') (float32), b2 = 0.2,
    gamma = 1.  There are no trained weights to load; these only give the
    projection its shape and a spread of outputs."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 31])))
    h = bf16_bits(rng.standard_normal((N, k, H), dtype=np.float32))
    w1 = bf16_bits(rng.standard_normal((Hp, H), dtype=np.float32) * np.float32(2.0 / np.sqrt(H)))
    b1 = (rng.standard_normal(Hp, dtype=np.float32) * np.float32(0.3)).astype(np.float32)
    w2 = (rng.standard_normal(Hp, dtype=np.float32) * np.float32(2.0 / np.sqrt(Hp))).astype(np.float32)
    return dict(hidden=h, w1=w1, b1=b1, w2=w2, b2=0.2, gamma=1.0)
