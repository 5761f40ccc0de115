"""Seeded synthetic workloads for the P-EAGLE parallel-draft step.

This module only draws numbers and lays them out; it holds none of the step's
arithmetic.  The CPU oracle tests, the GPU parity tests and the benchmark all
take their inputs from here, so both sides of every comparison see the same
bytes.

Shapes and value distributions follow the workloads the P-EAGLE pages describe:
GPT-OSS-20B-shaped and Llama-3.1-8B-shaped one-layer drafters fed by three
captured target hidden streams (the Qwen3-8B P-EAGLE drafter in "[RFC]: Add
random anchor for p-eagle first position" has three auxiliary verifier hidden
inputs), K = 7 draft depth at concurrency 1 and 64 ("P-EAGLE: parallel
speculative decoding in vLLM", performance benchmarks), and the stream RMS
values of "Attention Drift", Table 1 (Llama 3.1 8B row: 0.56, 0.58, 0.78).

Draw order.  Every tensor has a fixed name; the generator for a tensor is
``PCG64(SeedSequence(seed, spawn_key=(NAME_INDEX[name], chunk)))`` where the
tensor is drawn in chunks of ``CHUNK`` values.  Chunks are independent streams,
so a tensor can be filled by several threads and the bytes do not depend on the
thread count.  bf16 tensors are drawn in float32 and rounded to the nearest
bf16 (ties to even); they are returned as ``uint16`` bit patterns.
"""

from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 22

NAME_INDEX = {
    "batch": 0,
    "hidden": 1,
    "emb": 2,
    "emb_mask": 3,
    "h_shared": 4,
    "w_fc": 5,
    "w_qkv": 6,
    "w_o": 7,
    "w_gate": 8,
    "w_up": 9,
    "w_down": 10,
    "w_lm": 11,
    "k_cache": 12,
    "v_cache": 13,
    "verify_logits": 14,
    "verify_plan": 15,
    "attn_sink": 16,
    "cod_spans": 17,
    "cod_draws": 18,
}


@dataclasses.dataclass(frozen=True)
class Dims:
    """Drafter and step dimensions (one decoder layer, three target streams)."""

    d: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    inter: int
    vocab: int
    K: int
    block_size: int
    mask_id: int = 0
    post_norm: bool = False
    dtype: str = "bf16"  # "bf16" or "f32"
    eps: float = 1e-6
    rope_theta: float = 10000.0
    n_streams: int = 3
    n_layers: int = 1

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclasses.dataclass(frozen=True)
class Workload:
    """A step workload: dims plus the recipe of one ragged batch."""

    name: str
    dims: Dims
    batch: int
    # previous verify rows per request (n_r); an int or a per-request tuple
    n_prev: object
    # context lengths c_r: a tuple, or ("uniform", lo, hi) inclusive
    ctx: object
    # accepted counts a_r: "uniform" draws U[0, n_r - 1]; or a per-request tuple
    accepted: object = "uniform"
    stream_std: tuple = (1.0, 4.0, 16.0)
    weight_std: float = 0.02
    token_lo: int = 0
    seed: int = 0
    permute_blocks: bool = True
    spare_blocks: int = 0
    has_drafter: bool = True
    # per-head attention sink logits (GPT-oss attention), N(0, 1), float32
    sinks: bool = False
    description: str = ""

    def n_prev_list(self):
        if isinstance(self.n_prev, int):
            return [self.n_prev] * self.batch
        assert len(self.n_prev) == self.batch
        return list(self.n_prev)


def _gpt_oss_dims(post_norm=False):
    return Dims(d=2880, n_heads=64, n_kv_heads=8, head_dim=64, inter=7680,
                vocab=201088, K=7, block_size=16, post_norm=post_norm)


WORKLOADS = {
    # tiny fp32 step: the configuration the oracle checks row by row at 1e-5
    "tiny_fp32": Workload(
        name="tiny_fp32",
        dims=Dims(d=64, n_heads=4, n_kv_heads=2, head_dim=16, inter=128, vocab=512,
                  K=4, block_size=4, dtype="f32"),
        batch=2, n_prev=5, ctx=(16, 24), stream_std=(0.5, 1.0, 2.0), token_lo=1,
        description="tiny fp32 step, B=2, ctx 16/24, K=4, d=64, 4q/2kv heads of 16, I=128, V=512"),
    # metadata + hidden-state preparation only (no drafter weights but the embedding)
    "meta_prep_b64": Workload(
        name="meta_prep_b64",
        dims=Dims(d=2880, n_heads=64, n_kv_heads=8, head_dim=64, inter=7680,
                  vocab=201088, K=7, block_size=16),
        batch=64, n_prev=8, ctx=("uniform", 128, 8192), has_drafter=False,
        description="metadata + hidden-state prep, B=64, K=7, 3 streams of 2880 bf16"),
    "gptoss_b1_k7": Workload(
        name="gptoss_b1_k7", dims=_gpt_oss_dims(), batch=1, n_prev=8, ctx=(2048,),
        description="GPT-OSS-20B-shaped drafter, bf16, B=1, K=7, context 2048"),
    "gptoss_b64_k7_postnorm": Workload(
        name="gptoss_b64_k7_postnorm", dims=_gpt_oss_dims(post_norm=True), batch=64,
        n_prev=8, ctx=("uniform", 512, 8192),
        description="GPT-OSS-20B-shaped drafter, bf16, B=64, K=7, ctx U[512,8192], post-norm"),
    # the GPT-oss attention: per-head sink logits
    "gptoss_b64_k7_postnorm_sinks": Workload(
        name="gptoss_b64_k7_postnorm_sinks", dims=_gpt_oss_dims(post_norm=True), batch=64,
        n_prev=8, ctx=("uniform", 512, 8192), sinks=True,
        description="GPT-OSS-20B-shaped drafter with attention sinks, bf16, B=64, K=7, "
                    "ctx U[512,8192], post-norm"),
    # four decoder layers (every layer but the last over all non-rejected rows)
    "gptoss_b1_k7_4layers": Workload(
        name="gptoss_b1_k7_4layers", dims=dataclasses.replace(_gpt_oss_dims(), n_layers=4),
        batch=1, n_prev=8, ctx=(2048,),
        description="GPT-OSS-20B-shaped 4-layer drafter, bf16, B=1, K=7, context 2048"),
    "gptoss_b64_k7_postnorm_4layers": Workload(
        name="gptoss_b64_k7_postnorm_4layers",
        dims=dataclasses.replace(_gpt_oss_dims(post_norm=True), n_layers=4), batch=64,
        n_prev=8, ctx=("uniform", 512, 8192),
        description="GPT-OSS-20B-shaped 4-layer drafter, bf16, B=64, K=7, ctx U[512,8192], post-norm"),
    "llama8b_b32_k8_32k": Workload(
        name="llama8b_b32_k8_32k",
        dims=Dims(d=4096, n_heads=32, n_kv_heads=8, head_dim=128, inter=14336,
                  vocab=128256, K=8, block_size=16),
        batch=32, n_prev=9, ctx=(32768,) * 32, stream_std=(0.56, 0.58, 0.78),
        description="Llama-3.1-8B-shaped drafter, bf16, B=32, K=8, context 32768"),
    # small bf16 cases the oracle finishes in well under a second on every row;
    # every GEMM dimension spans several 128-row tiles plus a ragged tail
    "small_prenorm": Workload(
        name="small_prenorm",
        dims=Dims(d=320, n_heads=8, n_kv_heads=2, head_dim=64, inter=384, vocab=1000,
                  K=5, block_size=16),
        batch=3, n_prev=6, ctx=(37, 150, 260), stream_std=(1.0, 4.0, 16.0),
        description="small pre-norm bf16 step, hd 64"),
    "small_postnorm_hd128": Workload(
        name="small_postnorm_hd128",
        dims=Dims(d=256, n_heads=4, n_kv_heads=2, head_dim=128, inter=640, vocab=777,
                  K=8, block_size=16, post_norm=True),
        batch=4, n_prev=(9, 3, 1, 9), ctx=(0, 17, 100, 300), stream_std=(0.56, 0.58, 0.78),
        description="small post-norm bf16 step, hd 128, ragged n_r, a zero context"),
}


def get(name: str, **overrides) -> Workload:
    wl = WORKLOADS[name]
    if overrides:
        dims_over = {k: v for k, v in overrides.items() if k in Dims.__dataclass_fields__}
        wl_over = {k: v for k, v in overrides.items() if k not in dims_over}
        if dims_over:
            wl_over["dims"] = dataclasses.replace(wl.dims, **dims_over)
        wl = dataclasses.replace(wl, **wl_over)
    return wl


# ---------------------------------------------------------------------------
# random streams


def _seq(seed: int, name: str, chunk: int, layer: int = 0) -> np.random.Generator:
    # a later layer's tensor of the same name draws from its own stream
    key = (NAME_INDEX[name], chunk) if layer == 0 else (NAME_INDEX[name], chunk, layer)
    ss = np.random.SeedSequence(seed, spawn_key=key)
    return np.random.Generator(np.random.PCG64(ss))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(seed: int, name: str, n: int, std: float = 1.0, out=None, layer: int = 0) -> np.ndarray:
    """n float32 draws from N(0, std^2), chunked as described in the module doc."""
    out = np.empty(n, dtype=np.float32) if out is None else out
    n_chunks = (n + CHUNK - 1) // CHUNK

    def fill(c):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        g = _seq(seed, name, c, layer)
        g.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)

    if n_chunks <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    out = np.empty(u.shape, dtype=np.uint16)
    flat_u, flat_o = u.reshape(-1), out.reshape(-1)
    n = flat_u.size

    def conv(c):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        v = flat_u[lo:hi]
        r = (v + np.uint32(0x7FFF) + ((v >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        flat_o[lo:hi] = r.astype(np.uint16)

    n_chunks = (n + CHUNK - 1) // CHUNK
    if n_chunks <= 1:
        for c in range(n_chunks):
            conv(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(conv, range(n_chunks)))
    return out


def draw(seed: int, name: str, shape, std: float, dtype: str, layer: int = 0) -> np.ndarray:
    """A tensor of N(0, std^2) values in the workload dtype (f32, or bf16 bits)."""
    n = int(np.prod(shape))
    v = normal_f32(seed, name, n, std, layer=layer)
    if dtype == "bf16":
        return f32_to_bf16_bits(v).reshape(shape)
    return v.reshape(shape)


# ---------------------------------------------------------------------------
# one ragged batch


def make_batch(wl: Workload) -> dict:
    """Host arrays describing one ragged batch (the step's non-weight inputs).

    Returns qsl[B+1] i32, prev_tok[T_in] i32, prev_pos[T_in] i64, accepted[B] i32,
    bonus[B] i32, ctx[B] i64, block_table[B][MB] i32 (-1 past each request's
    blocks), num_blocks, and H_tgt[T_in][3][d] (f32, or bf16 bits).
    """
    dm = wl.dims
    g = _seq(wl.seed, "batch", 0)
    B = wl.batch
    n_prev = np.array(wl.n_prev_list(), dtype=np.int64)
    assert (n_prev >= 1).all()
    if isinstance(wl.ctx, tuple) and len(wl.ctx) == 3 and wl.ctx[0] == "uniform":
        ctx = g.integers(wl.ctx[1], wl.ctx[2] + 1, size=B).astype(np.int64)
    else:
        ctx = np.array(wl.ctx, dtype=np.int64)
        assert ctx.shape == (B,)
    if isinstance(wl.accepted, str):
        assert wl.accepted == "uniform"
        accepted = np.array([g.integers(0, n) for n in n_prev], dtype=np.int32)
    else:
        accepted = np.array(wl.accepted, dtype=np.int32)
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(n_prev)
    T_in = int(qsl[-1])
    prev_tok = g.integers(wl.token_lo, dm.vocab, size=T_in).astype(np.int32)
    bonus = g.integers(wl.token_lo, dm.vocab, size=B).astype(np.int32)
    prev_pos = np.concatenate([c + np.arange(n) for c, n in zip(ctx, n_prev)]).astype(np.int64)
    bs, K = dm.block_size, dm.K
    # blocks cover every position this step can write: up to c_r + n_r + K - 2
    n_blk = [(int(c) + int(n) + K - 1 + bs - 1) // bs for c, n in zip(ctx, n_prev)]
    MB = max(n_blk)
    num_blocks = int(sum(n_blk)) + wl.spare_blocks
    ids = g.permutation(num_blocks) if wl.permute_blocks else np.arange(num_blocks)
    block_table = np.full((B, MB), -1, dtype=np.int32)
    o = 0
    for r in range(B):
        block_table[r, : n_blk[r]] = ids[o : o + n_blk[r]]
        o += n_blk[r]
    hid = np.empty((T_in, dm.n_streams, dm.d), dtype=np.float32)
    raw = normal_f32(wl.seed, "hidden", T_in * dm.n_streams * dm.d).reshape(T_in, dm.n_streams, dm.d)
    for s in range(dm.n_streams):
        hid[:, s, :] = raw[:, s, :] * np.float32(wl.stream_std[s])
    H_tgt = f32_to_bf16_bits(hid) if dm.dtype == "bf16" else hid
    return dict(qsl=qsl, prev_tok=prev_tok, prev_pos=prev_pos, accepted=accepted,
                bonus=bonus, ctx=ctx, block_table=block_table, num_blocks=num_blocks,
                H_tgt=H_tgt, T_in=T_in, B=B)


def make_weights(wl: Workload, only=None) -> dict:
    """Drafter parameters.  Linear and embedding matrices, emb(mask) and h_shared
    are N(0, weight_std^2); RMSNorm gains are 1.  Layouts (row-major):
    emb[V][d], emb_mask[d], h_shared[d], gamma_stream[3][d], w_fc[d][4d],
    gamma_in[d], w_qkv[(H+2G)hd][d] (q heads, then k heads, then v heads),
    w_o[d][H hd], gamma_post[d], w_gate[I][d], w_up[I][d], w_down[d][I],
    gamma_final[d], w_lm[V][d]; with sinks, attn_sink[H] (float32 in both modes).
    With n_layers = N > 1, "layers" lists N - 1 dicts of the later layers' w_qkv,
    w_o, w_gate, w_up, w_down, gains (and sinks)."""
    dm, s, dt = wl.dims, wl.weight_std, wl.dims.dtype
    d, I, V = dm.d, dm.inter, dm.vocab
    shapes = {
        "emb": (V, d), "emb_mask": (d,), "h_shared": (d,),
        "w_fc": (d, 4 * d), "w_qkv": (dm.qkv_rows, d), "w_o": (d, dm.n_heads * dm.head_dim),
        "w_gate": (I, d), "w_up": (I, d), "w_down": (d, I), "w_lm": (V, d),
    }
    if not wl.has_drafter:
        shapes = {k: shapes[k] for k in ("emb", "emb_mask", "h_shared")}
    w = {}
    for name, shp in shapes.items():
        if only is not None and name not in only:
            continue
        w[name] = draw(wl.seed, name, shp, s, dt)
    one = np.float32(1.0)
    ones = (lambda shp: f32_to_bf16_bits(np.full(shp, one, np.float32))) if dt == "bf16" else \
        (lambda shp: np.full(shp, one, np.float32))
    w["gamma_stream"] = ones((dm.n_streams, d))
    if wl.has_drafter:
        for gname in ("gamma_in", "gamma_post", "gamma_final"):
            w[gname] = ones((d,))
        if wl.sinks:
            w["attn_sink"] = normal_f32(wl.seed, "attn_sink", dm.n_heads)
        # layers 2..N: the same recipe, each from its own streams
        if dm.n_layers > 1:
            w["layers"] = []
            for li in range(1, dm.n_layers):
                lw = {name: draw(wl.seed, name, shapes[name], s, dt, layer=li)
                      for name in ("w_qkv", "w_o", "w_gate", "w_up", "w_down")}
                for gname in ("gamma_in", "gamma_post", "gamma_final"):
                    lw[gname] = ones((d,))
                if wl.sinks:
                    lw["attn_sink"] = normal_f32(wl.seed, "attn_sink", dm.n_heads, layer=li)
                w["layers"].append(lw)
    return w


def make_kv_cache(wl: Workload, num_blocks: int) -> tuple:
    """Paged K and V caches [num_blocks][G][bs][hd] (one layer) or
    [N][num_blocks][G][bs][hd] (N layers), prior contents N(0, 1)."""
    dm = wl.dims
    shp = (num_blocks, dm.n_kv_heads, dm.block_size, dm.head_dim)
    if dm.n_layers <= 1:
        return (draw(wl.seed, "k_cache", shp, 1.0, dm.dtype),
                draw(wl.seed, "v_cache", shp, 1.0, dm.dtype))
    return tuple(np.stack([draw(wl.seed, name, shp, 1.0, dm.dtype, layer=li)
                           for li in range(dm.n_layers)]) for name in ("k_cache", "v_cache"))


# ---------------------------------------------------------------------------
# greedy verification batches


@dataclasses.dataclass(frozen=True)
class VerifyWorkload:
    """A verify batch: the target's logits over every verify row of a ragged
    batch, plus the row tokens (the last committed token, then the drafts)."""

    name: str
    batch: int
    # verify rows per request (n_r = K + 1 for K drafts); an int or a tuple
    n_rows: object
    vocab: int
    dtype: str = "f32"  # logits dtype: "f32" or "bf16"
    # fraction of rows whose greatest logit is planted at two indices
    tie_frac: float = 0.0
    seed: int = 0
    description: str = ""

    def n_rows_list(self):
        if isinstance(self.n_rows, int):
            return [self.n_rows] * self.batch
        assert len(self.n_rows) == self.batch
        return list(self.n_rows)


VERIFY_WORKLOADS = {
    # K = 7 drafts per request (8 verify rows) against a GPT-OSS-20B-sized vocabulary
    "verify_b64_k7": VerifyWorkload(
        name="verify_b64_k7", batch=64, n_rows=8, vocab=201088, dtype="f32", tie_frac=0.05,
        description="greedy verification of K=7 drafts, B=64, V=201088, fp32 logits"),
    "verify_b64_k7_bf16": VerifyWorkload(
        name="verify_b64_k7_bf16", batch=64, n_rows=8, vocab=201088, dtype="bf16",
        tie_frac=0.05,
        description="greedy verification of K=7 drafts, B=64, V=201088, bf16 logits"),
    "verify_b1_k7": VerifyWorkload(
        name="verify_b1_k7", batch=1, n_rows=8, vocab=201088, dtype="f32", tie_frac=0.0,
        description="greedy verification of K=7 drafts, B=1, V=201088, fp32 logits"),
    # small ragged cases: rows of 1001 fp32 / 777 bf16 logits start off the
    # 16-byte grid, one request has no drafts
    "verify_small": VerifyWorkload(
        name="verify_small", batch=5, n_rows=(8, 1, 3, 8, 2), vocab=1001, dtype="f32",
        tie_frac=0.3, description="small ragged verify batch, V=1001, fp32 logits"),
    "verify_small_bf16": VerifyWorkload(
        name="verify_small_bf16", batch=4, n_rows=(9, 2, 1, 5), vocab=777, dtype="bf16",
        tie_frac=0.3, description="small ragged verify batch, V=777, bf16 logits"),
}

# every drawn logit lies in [-LOGIT_CLIP, LOGIT_CLIP]; the planted greatest
# logit of a row is PLANTED_MAX, exact in fp32 and bf16
LOGIT_CLIP = 8.0
PLANTED_MAX = 9.0


def get_verify(name: str, **overrides) -> VerifyWorkload:
    wl = VERIFY_WORKLOADS[name]
    return dataclasses.replace(wl, **overrides) if overrides else wl


def make_verify_batch(wl: VerifyWorkload) -> dict:
    """Host arrays of one verify batch, with the target's greedy tokens and the
    accepted counts planted by construction.

    Logits are N(0, 1) clipped to [-8, 8]; each row's greatest logit (9.0) is
    planted at a uniform index g (and, in a tie_frac share of rows, also at a
    second, larger index, so the lowest-index rule picks g).  Per request a
    planted count a* ~ U[0, n_r - 1]: drafts 1..a* copy the planted tokens of
    the rows before them, draft a*+1 differs from its row's planted token, and
    the other tokens are uniform.

    Returns qsl[B+1] i32, tok[T_in] i32, logits[T_in][V] (f32, or bf16 bits),
    planted_target[T_in] i32, planted_accepted[B] i32, T_in, B, V.
    """
    n_rows = np.array(wl.n_rows_list(), dtype=np.int64)
    B, V = wl.batch, wl.vocab
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(n_rows)
    T_in = int(qsl[-1])
    g = _seq(wl.seed, "verify_plan", 0)
    logits = normal_f32(wl.seed, "verify_logits", T_in * V).reshape(T_in, V)
    np.clip(logits, -LOGIT_CLIP, LOGIT_CLIP, out=logits)
    target = g.integers(0, V, size=T_in).astype(np.int32)
    tie = g.random(T_in) < wl.tie_frac
    rows = np.arange(T_in)
    logits[rows, target] = PLANTED_MAX
    for i in np.nonzero(tie & (target < V - 1))[0]:
        logits[i, g.integers(int(target[i]) + 1, V)] = PLANTED_MAX
    tok = g.integers(0, V, size=T_in).astype(np.int32)
    accepted = np.zeros(B, dtype=np.int32)
    for r in range(B):
        q0, n = int(qsl[r]), int(n_rows[r])
        if n == 0:
            continue
        a = int(g.integers(0, n))
        accepted[r] = a
        tok[q0 + 1: q0 + 1 + a] = target[q0: q0 + a]
        if a + 1 < n:
            tok[q0 + a + 1] = (int(target[q0 + a]) + 1 + int(g.integers(0, V - 1))) % V
    out = f32_to_bf16_bits(logits) if wl.dtype == "bf16" else logits
    return dict(qsl=qsl, tok=tok, logits=out, planted_target=target,
                planted_accepted=accepted, T_in=T_in, B=B, V=V)


# ---------------------------------------------------------------------------
# COD training indices ("[RFC]: Add random anchor for p-eagle first position")


@dataclasses.dataclass(frozen=True)
class CodWorkload:
    """A batch of training sequences for the COD index and mask generator.

    Each sequence alternates spans with loss_mask 0 (prompt turns) and 1
    (response turns), so a large share of positions carries no loss, as the
    page's motivation says.  n_depth COD depths (depth 0 = every anchor),
    retain = the share of a depth's chains that reach the next (the page's
    "drop rate"), max_anchors = cap on depth-0 anchors (0 = no cap)."""

    name: str
    batch: int
    seq_len: object          # int or tuple of per-sequence lengths
    s_max: int               # row stride of the per-sequence arrays
    n_depth: int
    retain: float
    max_anchors: int
    prompt_span: tuple = (64, 512)
    response_span: tuple = (128, 1024)
    seed: int = 0
    description: str = ""

    def lens(self):
        if isinstance(self.seq_len, int):
            return [self.seq_len] * self.batch
        assert len(self.seq_len) == self.batch
        return list(self.seq_len)


COD_WORKLOADS = {
    # the page's 8K runs: max_anchors = 1024, drop rate 0.5, depths d0..d7
    "cod_s8192_a1024": CodWorkload(
        name="cod_s8192_a1024", batch=16, seq_len=8192, s_max=8192, n_depth=8, retain=0.5,
        max_anchors=1024,
        description="COD indices + asymmetric mask, 16 sequences x 8192, max_anchors 1024, "
                    "retain 0.5, 8 depths"),
    # the uncapped baseline of the page's 4K runs: every loss position is an anchor
    "cod_s4096_nocap": CodWorkload(
        name="cod_s4096_nocap", batch=8, seq_len=4096, s_max=4096, n_depth=5, retain=0.7,
        max_anchors=0,
        description="COD indices + asymmetric mask, 8 sequences x 4096, no anchor cap, "
                    "retain 0.7, 5 depths"),
    # small ragged cases: an empty sequence, a one-token one, lengths off every tile
    "cod_small": CodWorkload(
        name="cod_small", batch=6, seq_len=(3001, 0, 1, 777, 2048, 1500), s_max=3072, n_depth=8,
        retain=0.5, max_anchors=256, prompt_span=(16, 200), response_span=(32, 400),
        description="small ragged COD batch, max_anchors 256, retain 0.5, 8 depths"),
    "cod_tiny": CodWorkload(
        name="cod_tiny", batch=4, seq_len=(37, 64, 5, 50), s_max=64, n_depth=4, retain=0.7,
        max_anchors=8, prompt_span=(2, 9), response_span=(3, 12),
        description="tiny COD batch, max_anchors 8, retain 0.7, 4 depths"),
}


def get_cod(name: str, **overrides) -> CodWorkload:
    wl = COD_WORKLOADS[name]
    return dataclasses.replace(wl, **overrides) if overrides else wl


def make_cod_batch(wl: CodWorkload) -> dict:
    """Host arrays of one COD batch.

    loss_mask[B][s_max] u8: per sequence, spans alternate prompt (0) and response
    (1), lengths uniform in prompt_span / response_span, starting with a prompt
    span; positions past the sequence's length are 0.  u_anchor[B][s_max] and
    u_keep[B][n_depth-1][s_max]: float32 uniform in [0, 1) (the method's random
    draws).  seq_len[B] i32."""
    B, S, D = wl.batch, wl.s_max, wl.n_depth
    lens = np.array(wl.lens(), dtype=np.int32)
    assert lens.max(initial=0) <= S
    g = _seq(wl.seed, "cod_spans", 0)
    loss_mask = np.zeros((B, S), dtype=np.uint8)
    for b in range(B):
        pos, on = 0, 0
        while pos < lens[b]:
            lo, hi = wl.response_span if on else wl.prompt_span
            n = int(g.integers(lo, hi + 1))
            loss_mask[b, pos:min(pos + n, lens[b])] = on
            pos += n
            on ^= 1
    d = _seq(wl.seed, "cod_draws", 0)
    u_anchor = d.random((B, S), dtype=np.float32)
    u_keep = d.random((B, max(D - 1, 0), S), dtype=np.float32)
    return dict(seq_len=lens, loss_mask=loss_mask, u_anchor=u_anchor, u_keep=u_keep,
                B=B, S_max=S, n_depth=D, retain=wl.retain, max_anchors=wl.max_anchors)
