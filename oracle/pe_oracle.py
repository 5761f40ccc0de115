"""CPU oracle of the P-EAGLE parallel-draft step.  TEST INFRASTRUCTURE ONLY.

This module states, in plain fp64 numpy, what one parallel-draft step computes.
It exists to check the CUDA path.  Only the tests, the package's smoke check and
the benchmark's CPU-baseline leg may import it; the library never does, and it
shares no code with the CUDA sources (the seeded input generators are the only
thing both sides use, and they hold none of this arithmetic).

Sources (the pages this restates):
  [vLLM]  "P-EAGLE: parallel speculative decoding in vLLM" (agentlenshq blog,
          zh-TW and Korean editions): "Architecture and mechanism", step 2
          "Parallel drafting" (prompt-position pairing shifted by one, the NTP
          position, the MTP positions 2..K with the learned emb(mask) and
          h_shared, one pass through the layers and LM head); "vLLM
          implementation details": "Fused Triton kernel" (the batch metadata),
          "Hidden-state management" (the copy / broadcast kernel), "KV cache and
          CUDA graphs" (rejected tokens map to PADDING_SLOT_ID = -1).
  [Drift] "Attention Drift: what autoregressive speculative decoding models
          learn": section 2 (EAGLE-3 feeds the fused target hidden states through
          an fc projection into one pre-norm decoder layer), section 4.1 (RMS is
          ||x||_2 / sqrt(d)), Observation 2 (an RMSNorm on each captured target
          stream before the fc), abstract and section 1 (post-norm drafter);
          section 2 also states verification: the target scores the drafts in
          one pass and keeps the longest prefix it accepts (verify_greedy).
  [RFC]   "[RFC]: Add random anchor for p-eagle first position": the P-EAGLE
          drafter is one transformer layer fed by three auxiliary verifier hidden
          streams.

Readings where the pages are silent (each one is listed in the design notes):
  * K-1 MASK rows per request, appended after the request's n_r copied rows;
    rejected rows stay in place with is_rejected = 1 and slot = -1.
  * A copied row j takes token prev_tok[j+1]; the NTP row j = a_r takes the bonus
    token b_r; the last copied row, when rejected, also takes b_r.
  * MASK row m (m = 1..K-1) sits at position prev_pos[a_r] + m and writes its KV.
  * h_shared has width d and fills all three stream slots; emb(mask) is its own
    learned vector, chosen by is_masked.
  * Concatenation order [h_low, h_mid, h_high, emb]; no biases anywhere.
  * RMSNorm(x) = x * gamma / sqrt(mean(x^2) + eps).
  * RoPE: rotate-half pairing (i, i + hd/2), inverse frequency theta^(-2i/hd).
  * Attention scale 1/sqrt(hd); query head h reads KV head floor(h / (H/G)).
  * Optional per-head sink logits (float32 in both modes): one more logit in
    each head's softmax with a zero value row.
  * Pre-norm layer: u = RMSNorm(x; gamma_in); a = x + O(attn);
    y = a + MLP(RMSNorm(a; gamma_post)); z = RMSNorm(y; gamma_final).
    Post-norm layer: u = x; a = RMSNorm(x + O(attn); gamma_post);
    z = RMSNorm(a + MLP(a); gamma_final), no further norm.
  * MLP is SwiGLU: down(silu(gate(m)) * up(m)), silu(t) = t / (1 + e^-t).
  * Greedy draft: argmax of the logits, lowest index on ties.
  * bf16 mode (weights and the KV cache in bf16): a value is rounded to bf16
    (nearest, ties to even) only where the step stores it as a bf16 tensor:
    the drafter input A, q/k/v after RoPE (the cache dtype), the attention
    output and z.  Every other intermediate (the fc output x, the QKV operand u,
    the MLP input, the SwiGLU product, the residual sums, a layer's output
    passed to the next) is kept exact (fp64): the reading is that nothing is
    rounded where the pages fix no storage type.  Logits stay unrounded.  fp32
    mode rounds nothing (fp64 throughout).

Pins: every function here is checked in tests/test_oracle_*.py against closed
forms, brute force or invariants the pages fix.  The end-to-end logits beyond
those invariants are "parity unpinned": the pages print no worked example of
the step.
"""

from __future__ import annotations

import numpy as np

PADDING_SLOT_ID = -1


# ---------------------------------------------------------------------------
# number formats


def bf16_round(x):
    """Nearest bf16 value (ties to even) of fp64 values, returned as fp64.

    bf16 keeps 8 significant bits.  frexp writes x = m * 2^e with 0.5 <= |m| < 1,
    so m * 2^8 lies in [128, 256) and rounding it to an integer (rint rounds
    halves to even) keeps exactly 8 bits.  The bf16 subnormal and overflow
    ranges are not modelled (no value of the step comes near them).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_decode(bits):
    """uint16 bf16 bit patterns -> fp64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def decode(arr, dtype):
    """A stored tensor (float32, or bf16 bits) as fp64."""
    if dtype == "bf16":
        return bf16_decode(arr)
    return np.asarray(arr, dtype=np.float64)


def _rounder(dtype):
    return bf16_round if dtype == "bf16" else (lambda v: np.asarray(v, dtype=np.float64))


def _exact(v):
    """An intermediate the step does not store as a bf16 tensor: kept in fp64."""
    return np.asarray(v, dtype=np.float64)


# ---------------------------------------------------------------------------
# step (1): batch metadata   [vLLM] "Fused Triton kernel", "KV cache and CUDA graphs",
#                            "Parallel drafting"


def slot_of(block_table, r, pos, block_size):
    """Cache slot of position pos of request r: physical block * bs + offset."""
    return int(block_table[r][pos // block_size]) * block_size + pos % block_size


def prepare_metadata(qsl, prev_tok, prev_pos, accepted, bonus, block_table, K, mask_id,
                     block_size):
    """Build the drafter batch from the previous verify batch.

    Request r owns input rows qsl[r]..qsl[r+1]-1 (n_r rows) and accepted a_r of
    them past the first (0 <= a_r <= n_r - 1).  Its output rows are its n_r
    copied rows followed by K-1 MASK rows:
      copied row j < a_r : token prev_tok[j+1], position prev_pos[j], hidden from
                           input row j (the prompt-position pairing, shifted by one)
      copied row j = a_r : the NTP row: bonus token b_r with the hidden state of
                           input row a_r (h_context)
      copied row j > a_r : rejected; token prev_tok[j+1] (b_r for the last row),
                           slot PADDING_SLOT_ID so no KV is written
      MASK row m=1..K-1  : token mask_id, position prev_pos[a_r] + m, no hidden
                           source (h_shared is used), is_masked = 1
    Non-rejected rows write KV at slot = block_table[r][pos // bs] * bs + pos % bs.
    The K sample rows (NTP row, then the MASK rows) predict draft tokens t_1..t_K.
    """
    qsl = np.asarray(qsl)
    B = len(accepted)
    T_in = int(qsl[B])
    T_out = T_in + B * (K - 1)
    out_qsl = np.zeros(B + 1, np.int32)
    valid_qsl = np.zeros(B + 1, np.int32)
    tok = np.zeros(T_out, np.int32)
    pos = np.zeros(T_out, np.int64)
    is_rejected = np.zeros(T_out, np.uint8)
    is_masked = np.zeros(T_out, np.uint8)
    hidden_src = np.zeros(T_out, np.int32)
    slot = np.zeros(T_out, np.int64)
    valid_rows = np.full(T_out, -1, np.int32)
    sample_idx = np.zeros(B * K, np.int32)
    seq_len = np.zeros(B, np.int32)
    o = 0
    nv = 0
    for r in range(B):
        out_qsl[r] = o
        valid_qsl[r] = nv
        base = int(qsl[r])
        n_r = int(qsl[r + 1]) - base
        a = int(accepted[r])
        assert 0 <= a <= n_r - 1, "accepted count out of range"
        for j in range(n_r):
            i = base + j
            if j == a:
                tok[o] = bonus[r]
            elif j < n_r - 1:
                tok[o] = prev_tok[i + 1]
            else:
                tok[o] = bonus[r]
            pos[o] = prev_pos[i]
            hidden_src[o] = i
            if j > a:
                is_rejected[o] = 1
                slot[o] = PADDING_SLOT_ID
            else:
                slot[o] = slot_of(block_table, r, int(pos[o]), block_size)
                valid_rows[nv] = o
                nv += 1
            if j == a:
                sample_idx[r * K] = o
            o += 1
        p0 = int(prev_pos[base + a])
        for m in range(1, K):
            tok[o] = mask_id
            pos[o] = p0 + m
            hidden_src[o] = -1
            is_masked[o] = 1
            slot[o] = slot_of(block_table, r, p0 + m, block_size)
            valid_rows[nv] = o
            nv += 1
            sample_idx[r * K + m] = o
            o += 1
        seq_len[r] = p0 + K
    out_qsl[B] = o
    valid_qsl[B] = nv
    return dict(out_qsl=out_qsl, tok=tok, pos=pos, is_rejected=is_rejected,
                is_masked=is_masked, hidden_src=hidden_src, slot=slot,
                valid_qsl=valid_qsl, valid_rows=valid_rows, n_valid=nv,
                sample_idx=sample_idx, seq_len=seq_len, T_out=T_out)


# ---------------------------------------------------------------------------
# step (2): hidden-state map and placeholder broadcast   [vLLM] "Hidden-state management",
#                                                        "Parallel drafting" (MTP positions)


def gather_hidden(meta, H_tgt, h_shared):
    """G[o][s] = H_tgt[hidden_src[o]][s] for copied rows, h_shared for MASK rows.

    H_tgt is [T_in][S][d] in fp64; h_shared is [d] and fills every stream slot.
    """
    T_out = meta["T_out"]
    S, d = H_tgt.shape[1], H_tgt.shape[2]
    G = np.empty((T_out, S, d))
    for o in range(T_out):
        src = int(meta["hidden_src"][o])
        G[o] = H_tgt[src] if src >= 0 else h_shared[None, :]
    return G


def embed_rows(meta, emb, emb_mask):
    """E[o] = emb(mask) for MASK rows, the token's embedding row otherwise.

    emb may be a callable mapping a token id to its fp64 row (for vocabularies
    too large to decode whole)."""
    T_out = meta["T_out"]
    rows = []
    for o in range(T_out):
        if meta["is_masked"][o]:
            rows.append(np.asarray(emb_mask, dtype=np.float64))
        else:
            t = int(meta["tok"][o])
            rows.append(emb(t) if callable(emb) else emb[t])
    return np.stack(rows) if rows else np.zeros((0, len(emb_mask)))


# ---------------------------------------------------------------------------
# step (3): drafter input   [Drift] section 4.1 (RMS), Observation 2; section 2 (fc fusion)


def rms(x):
    """Root mean square over the last axis: ||x||_2 / sqrt(d)."""
    x = np.asarray(x, dtype=np.float64)
    return np.sqrt(np.mean(x * x, axis=-1))


def rmsnorm(x, gamma, eps):
    """x * gamma / sqrt(mean(x^2) + eps) over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * gamma


def drafter_input(G, E, gamma_stream, eps, dtype):
    """A[o] = [RMSNorm(G[o][0]), RMSNorm(G[o][1]), RMSNorm(G[o][2]), E[o]], each
    stream with its own gain, concatenated along the feature axis."""
    R = _rounder(dtype)
    S = G.shape[1]
    parts = [rmsnorm(G[:, s, :], gamma_stream[s], eps) for s in range(S)]
    return R(np.concatenate(parts + [E], axis=-1))


# ---------------------------------------------------------------------------
# step (4): decoder layer pieces


def linear(x, W):
    """y = x W^T: x is [n][in], W is [out][in] (the row-major weight layout)."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def rope(x, pos, theta):
    """Rotary embedding, rotate-half pairing.

    x is [n][heads][hd]; pos is [n].  For i < hd/2 the pair (x_i, x_{i+hd/2}) is
    rotated by the angle pos * theta^(-2i/hd)."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def softmax(s):
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - s.max())
    return e / e.sum()


def attend(q, K_seq, V_seq, sink=None):
    """One query head over keys 0..n-1: softmax(K q / sqrt(hd)) weighted sum of V.

    q is [hd]; K_seq and V_seq are [n][hd].  sink (optional): the head's learned
    sink logit ("Attention Drift", section 3, the GPT-oss attention: a per-head
    bias logit in the softmax denominator, an explicit option to attend to
    nothing).  It joins the softmax as one more logit whose value row is zero,
    so the weights of the real keys sum to less than one."""
    hd = q.shape[-1]
    s = K_seq @ q / np.sqrt(hd)
    if sink is None:
        p = softmax(s)
    else:
        p = softmax(np.append(s, float(sink)))[:-1]
    return p @ V_seq


def silu(t):
    return t / (1.0 + np.exp(-t))


def swiglu_mlp(m, w_gate, w_up, w_down):
    """down(silu(gate(m)) * up(m))."""
    h = silu(linear(m, w_gate)) * linear(m, w_up)
    return linear(h, w_down)


def argmax_lowest(logits):
    """Greedy pick per row; ties go to the lowest index."""
    return np.argmax(logits, axis=-1).astype(np.int32)  # numpy returns the first maximum


# ---------------------------------------------------------------------------
# the whole step


class _Params:
    """fp64 views of the drafter parameters, decoded on first use."""

    def __init__(self, w, dtype):
        self._w, self._dt, self._cache = w, dtype, {}

    def __getitem__(self, name):
        if name not in self._cache:
            self._cache[name] = decode(self._w[name], self._dt)
        return self._cache[name]

    def raw(self, name):
        """A parameter as stored, or None when absent (the optional sink logits)."""
        return self._w.get(name)

    def emb_row(self, t):
        return decode(self._w["emb"][t], self._dt)

    def lm_logits(self, z, chunk=16384):
        """z W_lm^T, decoding W_lm a block of rows at a time."""
        W = self._w["w_lm"]
        V = W.shape[0]
        out = np.empty((z.shape[0], V))
        for v0 in range(0, V, chunk):
            out[:, v0:v0 + chunk] = z @ decode(W[v0:v0 + chunk], self._dt).T
        return out


def decoder_layer(dims, Pl, h_in, pos, att_rows, Kseq, Vseq, R, last):
    """One decoder layer over a request's rows.

    h_in: the layer's input rows [n][d] (fp64); pos: their positions.  Kseq,
    Vseq: the layer's cache of the request as position-indexed [L][G][hd]
    sequences, before this step; every row's k and v are written into them at
    its position ("KV cache and CUDA graphs": the cache is read after this
    step's writes).  att_rows: the rows whose attention, O and MLP are needed
    (all of them, or the sample rows of the last layer).  R: the rounding of
    the tensors the step stores in bf16.  [Drift] section 2: the EAGLE-3 drafter
    layer is a pre-norm decoder layer; abstract and section 1: the post-norm
    variant normalises after each residual.

    Returns u, q (all rows), k, v, attn, a (att_rows), y (the MLP residual sum),
    out (the layer's output: the next layer's input, or before z for the last
    layer: RMSNorm(y; gamma_final)) and hidden (the drafter's output hidden
    state: pre-norm y, post-norm the normalised output; both unrounded).
    """
    H, G_, hd = dims.n_heads, dims.n_kv_heads, dims.head_dim
    group = H // G_
    u = _exact(h_in) if dims.post_norm else rmsnorm(h_in, Pl["gamma_in"], dims.eps)
    qkv = linear(u, Pl["w_qkv"])
    q = qkv[:, : H * hd].reshape(-1, H, hd)
    k = qkv[:, H * hd: (H + G_) * hd].reshape(-1, G_, hd)
    v = qkv[:, (H + G_) * hd:].reshape(-1, G_, hd)
    q = R(rope(q, pos, dims.rope_theta))
    k = R(rope(k, pos, dims.rope_theta))
    v = R(v)
    for i, p in enumerate(pos):
        Kseq[int(p)] = k[i]
        Vseq[int(p)] = v[i]
    sinks = Pl.raw("attn_sink")
    attn = np.empty((len(att_rows), H, hd))
    for kk, i in enumerate(att_rows):
        n_keys = int(pos[i]) + 1      # causal: the full context plus earlier rows
        for h in range(H):
            g = h // group
            attn[kk, h] = attend(q[i, h], Kseq[:n_keys, g], Vseq[:n_keys, g],
                                 None if sinks is None else float(sinks[h]))
    attn = R(attn.reshape(len(att_rows), H * hd))
    xs = h_in[att_rows]
    o_proj = linear(attn, Pl["w_o"])
    if dims.post_norm:
        a = rmsnorm(xs + o_proj, Pl["gamma_post"], dims.eps)
        y = a + swiglu_mlp(a, Pl["w_gate"], Pl["w_up"], Pl["w_down"])
        # a post-norm layer's output is normalised (the last one's is z)
        out = rmsnorm(y, Pl["gamma_final"], dims.eps)
        hidden = out
    else:
        a = xs + o_proj
        m = rmsnorm(a, Pl["gamma_post"], dims.eps)
        y = a + swiglu_mlp(m, Pl["w_gate"], Pl["w_up"], Pl["w_down"])
        out = y if not last else rmsnorm(y, Pl["gamma_final"], dims.eps)
        hidden = y
    return dict(u=u, q=q, k=k, v=v, attn=attn, a=a, y=y, out=out, hidden=hidden)


def params(w, dtype):
    """fp64 views of stored drafter parameters (decoded on first use), the form
    autoregressive_pass takes."""
    return _Params(w, dtype)


def request_kv_sequence(cache, block_table, r, n_pos, block_size, dtype):
    """The first n_pos cache positions of request r as [n_pos][G][hd] fp64,
    read through its block table (cache is [num_blocks][G][bs][hd])."""
    nblk = (n_pos + block_size - 1) // block_size
    blocks = np.asarray(block_table[r][:nblk], dtype=np.int64)
    assert (blocks >= 0).all()
    seq = cache[blocks]                       # [nblk][G][bs][hd]
    seq = np.transpose(seq, (0, 2, 1, 3))     # [nblk][bs][G][hd]
    seq = seq.reshape(nblk * block_size, seq.shape[2], seq.shape[3])[:n_pos]
    return decode(seq, dtype)


def draft_step(dims, w, batch, k_cache=None, v_cache=None, requests=None, want_logits=True,
               round_stores=True):
    """One parallel-draft step.

    dims: object with d, n_heads, n_kv_heads, head_dim, inter, vocab, K,
          block_size, mask_id, post_norm, dtype, eps, rope_theta.
    w:    parameters as stored (float32 arrays, or bf16 bit patterns).  With
          dims.n_layers = N > 1, w["layers"] holds N - 1 dicts of the later
          layers' parameters (gamma_in, w_qkv, w_o, gamma_post, w_gate, w_up,
          w_down, gamma_final, optional attn_sink); the top-level ones are layer 1's.
    batch: qsl, prev_tok, prev_pos, accepted, bonus, block_table, H_tgt.
    k_cache, v_cache: paged caches [num_blocks][G][bs][hd] (one layer) or
          [N][num_blocks][G][bs][hd], as stored, before the step; they are read,
          never modified.
    requests: indices of the requests to run the layer for (default: all);
          metadata is always built for the whole batch.
    round_stores: in bf16 mode, round the tensors the step stores in bf16 (A,
          q/k/v, the attention output, z).  False computes the plain fp64
          definition on the same stored inputs (nothing rounded at all).

    Returns {"meta": ..., "req": {r: per-request results}} where a request's
    results hold, over its valid rows in order: rows, A, x, u, k, v, slot (u, k
    and v of the first layer) and k_layers, v_layers (every layer's); and over
    its K sample rows: q, attn, a (the last layer's), z, logits, draft.

    Layers ("P-EAGLE: parallel speculative decoding in vLLM", Parallel drafting:
    all positions pass through the N layers and the LM head).  Pre-norm: layer l
    maps x_l to x_{l+1} = a + MLP(RMSNorm(a)) with a = x_l + O(attn); the final
    norm (the last layer's gamma_final) gives z.  Post-norm: x_{l+1} =
    RMSNorm(a + MLP(a); gamma_final_l) with a = RMSNorm(x_l + O(attn)); the last
    layer's output is z.  Each layer has its own KV cache.
    """
    dt = dims.dtype
    R = _rounder(dt) if round_stores else _exact
    P = _Params(w, dt)
    K, H, G_, hd = dims.K, dims.n_heads, dims.n_kv_heads, dims.head_dim
    meta = prepare_metadata(batch["qsl"], batch["prev_tok"], batch["prev_pos"],
                            batch["accepted"], batch["bonus"], batch["block_table"],
                            K, dims.mask_id, dims.block_size)
    B = len(batch["accepted"])
    if requests is None:
        requests = range(B)
    H_tgt = batch["H_tgt"]
    h_shared = P["h_shared"]
    emb_mask = P["emb_mask"]
    gam_s = P["gamma_stream"]
    n_layers = max(1, int(getattr(dims, "n_layers", 1)))
    layer_params = [P] + [_Params(lw, dt) for lw in w.get("layers", [])[: n_layers - 1]]
    assert len(layer_params) == n_layers, "w['layers'] holds the layers after the first"
    out = {"meta": meta, "req": {}}
    for r in requests:
        v0, v1 = int(meta["valid_qsl"][r]), int(meta["valid_qsl"][r + 1])
        rows = meta["valid_rows"][v0:v1].astype(np.int64)
        # (2) hidden map + placeholders, (3) per-stream norm + concat
        Grows = np.stack([decode(H_tgt[meta["hidden_src"][o]], dt) if meta["hidden_src"][o] >= 0
                          else np.broadcast_to(h_shared, (dims.n_streams, dims.d))
                          for o in rows])
        Erows = np.stack([emb_mask if meta["is_masked"][o] else P.emb_row(int(meta["tok"][o]))
                          for o in rows])
        A = drafter_input(Grows, Erows, gam_s, dims.eps, dt if round_stores else "f32")
        # (4) fc, then the decoder layers.  Every layer but the last runs over all
        # the request's valid rows (the next layer's keys and values need them);
        # the last runs its attention, O and MLP over the K sample rows only
        # (the other rows' outputs are dead).
        x = linear(A, P["w_fc"])
        L = int(meta["seq_len"][r])
        pos = meta["pos"][rows]
        # sample rows are the last K valid rows of the request (NTP row, MASK rows)
        s_loc = np.arange(len(rows) - K, len(rows))
        assert (rows[s_loc] == meta["sample_idx"][r * K:(r + 1) * K]).all()
        h_in = x
        k_layers, v_layers = [], []
        for li, Pl in enumerate(layer_params):
            last = li == n_layers - 1
            # this layer's cache before this step, as a position-indexed sequence
            kc_l = k_cache if n_layers == 1 else k_cache[li]
            vc_l = v_cache if n_layers == 1 else v_cache[li]
            Kseq = request_kv_sequence(kc_l, batch["block_table"], r, L, dims.block_size, dt)
            Vseq = request_kv_sequence(vc_l, batch["block_table"], r, L, dims.block_size, dt)
            att_rows = s_loc if last else np.arange(len(rows))
            ly = decoder_layer(dims, Pl, h_in, pos, att_rows, Kseq, Vseq, R, last)
            if li == 0:
                u0 = ly["u"]
            k_layers.append(ly["k"])
            v_layers.append(ly["v"])
            q, attn, a = ly["q"], ly["attn"], ly["a"]
            h_in = ly["out"]
        z = R(h_in)
        res = dict(rows=rows, A=A, x=x, u=u0, k=k_layers[0], v=v_layers[0], slot=meta["slot"][rows],
                   q=q[s_loc], attn=attn, a=a, z=z, h=ly["hidden"], k_layers=k_layers,
                   v_layers=v_layers)
        if want_logits:
            logits = P.lm_logits(z)
            res["logits"] = logits
            res["draft"] = argmax_lowest(logits)
        out["req"][r] = res
    return out


def autoregressive_pass(dims, P, hidden_prev, token_prev, p, Kseq, Vseq, round_stores=True):
    """One pass k >= 2 of the autoregressive drafting for one request: the row at
    position p whose three stream slots hold hidden_prev (the drafter's hidden
    state of the pass before, [d]) and whose token is token_prev.  Its k and v
    are written into the request's cache sequences Kseq / Vseq at p (the cache
    the pass attends to after its write).  P: the parameters (_Params).
    Returns z, logits, draft, hidden (the state passed to the next pass), k, v."""
    dt = dims.dtype
    R = _rounder(dt) if round_stores else _exact
    G = np.broadcast_to(np.asarray(hidden_prev, np.float64), (dims.n_streams, dims.d))[None]
    A = drafter_input(G, P.emb_row(int(token_prev))[None], P["gamma_stream"], dims.eps,
                      dt if round_stores else "f32")
    x = linear(A, P["w_fc"])
    ly = decoder_layer(dims, P, x, np.array([p]), np.array([0]), Kseq, Vseq, R, True)
    z = R(ly["out"])
    lg = P.lm_logits(z)
    return dict(z=z[0], logits=lg[0], draft=int(argmax_lowest(lg)[0]), hidden=ly["hidden"][0],
                k=ly["k"][0], v=ly["v"][0])


def draft_autoregressive(dims, w, batch, k_cache, v_cache, requests=None, round_stores=True):
    """The autoregressive EAGLE-3 drafting that the parallel step replaces: K
    sequential passes of the same one-layer drafter, one draft token per pass.

    [vLLM] "Solving the autoregressive drafting bottleneck": K draft tokens cost
    K sequential forward passes of the drafter.  [Drift] section 3 and section
    4.1 (Table 1, Observation 3): once drafting starts, the drafter consumes its
    own hidden state instead of the target's.

      pass 1      the parallel step with K = 1: the request's non-rejected rows,
                  the NTP row (bonus token, target hidden state) as the one
                  sample row; it drafts t_1.
      pass k > 1  one row per request at position prev_pos[a_r] + k - 1 (the
                  position of P-EAGLE's MASK row k - 1): the drafter's hidden
                  state from pass k - 1 fills the three stream slots (where the
                  parallel step puts h_shared) and the embedding of t_{k-1} the
                  token slot; it drafts t_k.
    The hidden state passed on is the layer's output before the LM head's norm:
    y for a pre-norm layer, the normalised output for a post-norm layer (both
    unrounded).  Every pass writes its rows' KV and attends to the cache after
    its own write.  One decoder layer (dims.n_layers == 1).

    Returns {"meta": pass 1's metadata, "req": {r: dict(draft [K], logits [K][V],
    z [K][d], hidden [K][d], pos [K], first (pass 1's draft_step results),
    k_pass / v_pass [K-1][G][hd] (the KV passes 2..K write))}}.
    """
    assert max(1, int(getattr(dims, "n_layers", 1))) == 1, "one decoder layer"
    import dataclasses

    dt = dims.dtype
    P = _Params(w, dt)
    K = dims.K
    d1 = dataclasses.replace(dims, K=1)
    first = draft_step(d1, w, batch, k_cache, v_cache, requests=requests, round_stores=round_stores)
    meta = first["meta"]
    out = {"meta": meta, "req": {}}
    for r, r1 in first["req"].items():
        # the cache after pass 1: prior context plus the non-rejected rows' writes
        P0 = int(meta["pos"][meta["sample_idx"][r]])
        L = P0 + K
        Kseq = request_kv_sequence(k_cache, batch["block_table"], r, L, dims.block_size, dt)
        Vseq = request_kv_sequence(v_cache, batch["block_table"], r, L, dims.block_size, dt)
        for i, o in enumerate(r1["rows"]):
            Kseq[int(meta["pos"][o])] = r1["k"][i]
            Vseq[int(meta["pos"][o])] = r1["v"][i]
        drafts, logits, zs, hs, poss = [int(r1["draft"][0])], [r1["logits"][0]], [r1["z"][0]], \
            [r1["h"][0]], [P0]
        ks, vs = [], []
        for k in range(2, K + 1):
            p = P0 + k - 1
            one = autoregressive_pass(dims, P, hs[-1], drafts[-1], p, Kseq, Vseq, round_stores)
            drafts.append(one["draft"])
            logits.append(one["logits"])
            zs.append(one["z"])
            hs.append(one["hidden"])
            poss.append(p)
            ks.append(one["k"])
            vs.append(one["v"])
        out["req"][r] = dict(draft=np.array(drafts, np.int32), logits=np.stack(logits),
                             z=np.stack(zs), hidden=np.stack(hs), pos=np.array(poss, np.int64),
                             first=r1, k_pass=np.array(ks).reshape(-1, dims.n_kv_heads, dims.head_dim),
                             v_pass=np.array(vs).reshape(-1, dims.n_kv_heads, dims.head_dim))
    return out


def prepare_inputs(dims, w, batch):
    """Steps (1)-(3) over every output row: metadata, G, E and A (all T_out rows)."""
    dt = dims.dtype
    meta = prepare_metadata(batch["qsl"], batch["prev_tok"], batch["prev_pos"],
                            batch["accepted"], batch["bonus"], batch["block_table"],
                            dims.K, dims.mask_id, dims.block_size)
    H = decode(batch["H_tgt"], dt)
    G = gather_hidden(meta, H, decode(w["h_shared"], dt))
    E = embed_rows(meta, lambda t: decode(w["emb"][t], dt), decode(w["emb_mask"], dt))
    A = drafter_input(G, E, decode(w["gamma_stream"], dt), dims.eps, dt)
    return meta, G, E, A


# ---------------------------------------------------------------------------
# greedy verification (closes the loop into the next step's accepted counts
# and bonus tokens)


def target_argmax(logits):
    """Greedy token of each verify row: the index of the largest logit, lowest
    index on ties, a NaN counting as larger than every number (numpy's argmax
    rule: the first NaN wins).  -0.0 and +0.0 are equal.  Logits are decoded to
    fp64 first, which is exact for fp32 and bf16 inputs."""
    return np.argmax(np.asarray(logits, dtype=np.float64), axis=-1).astype(np.int32)


def verify_greedy(qsl, tok, logits):
    """Greedy verification of a ragged verify batch.

    "Attention Drift", section 2 (preliminaries): the target scores the drafted
    tokens in one forward pass and keeps the longest prefix its own
    distribution accepts.  The drafts here are greedy, so the target's
    distribution is read at temperature 0 and acceptance is exact agreement
    with the target's greedy token.

    Request r owns verify rows qsl[r] .. qsl[r+1]-1 (n_r of them).  Row 0 of a
    request carries the last committed token, row j >= 1 carries draft j, and
    logits[row] are the target's logits after that row's token.  So draft j is
    accepted when it equals the target's greedy token of row j-1 and every
    earlier draft was accepted; the bonus (correction) token is the target's
    greedy token right after the accepted prefix.

    Returns (target_tok[T_in] i32, accepted[B] i32, bonus[B] i32).  An empty
    request (n_r = 0) gets accepted 0 and bonus -1.
    """
    qsl = np.asarray(qsl, dtype=np.int64)
    tok = np.asarray(tok, dtype=np.int64)
    B = len(qsl) - 1
    target = target_argmax(logits) if len(tok) else np.zeros(0, np.int32)
    accepted = np.zeros(B, dtype=np.int32)
    bonus = np.full(B, -1, dtype=np.int32)
    for r in range(B):
        q0, n = int(qsl[r]), int(qsl[r + 1] - qsl[r])
        if n <= 0:
            continue
        a = 0
        while a + 1 < n and tok[q0 + a + 1] == target[q0 + a]:
            a += 1
        accepted[r] = a
        bonus[r] = target[q0 + a]
    return target, accepted, bonus
