/*
 * pe.h -- C-ABI of the P-EAGLE parallel-draft step on one GB300 (sm_103a).
 *
 * One parallel-draft step turns the previous verify batch of a ragged set of
 * requests into K draft tokens per request with a single drafter forward pass.
 * The calls below follow the problem statement of "P-EAGLE: parallel
 * speculative decoding in vLLM":
 *   pe_prepare_inputs  the fused batch-metadata build ("Fused Triton kernel":
 *                      copy previous token ids and positions, insert the bonus
 *                      token, fill the parallel-draft slots with the MASK id,
 *                      emit the rejected-token mask, the masked-token mask and
 *                      the hidden-state map; rejected tokens map to
 *                      PADDING_SLOT_ID = -1 per "KV cache and CUDA graphs"),
 *                      the hidden-state copy / h_shared broadcast
 *                      ("Hidden-state management") and the drafter input, which
 *                      applies an RMSNorm to each captured target stream
 *                      ("Attention Drift", section 4.1, Observation 2) and
 *                      concatenates them with the token embedding.
 *   pe_draft_step      the drafter pass ("Parallel drafting": all positions go
 *                      through the layer at once): fc projection, one decoder
 *                      layer (QKV, RoPE, paged KV write, paged attention over
 *                      the context plus earlier draft positions, SwiGLU MLP,
 *                      pre-norm or post-norm residuals) and the final norm.
 *   pe_argmax          the LM head fused with a per-row greedy argmax.
 *   pe_verify_greedy   the target's greedy verification of the drafts, which
 *                      yields the next step's accepted counts and bonus tokens.
 *   pe_draft_autoregressive
 *                      the K-pass autoregressive drafting the parallel step
 *                      replaces, on the same kernels (the baseline).
 *   pe_cod_sample_indices, pe_cod_mask
 *                      the training side's COD index lists and asymmetric
 *                      attention mask ("[RFC]: Add random anchor for p-eagle
 *                      first position").
 *
 * Conventions for every call
 *   - All tensor arguments are DEVICE pointers owned by the caller; the library
 *     never frees or keeps them past the call (weights excepted: pe_create
 *     borrows them for the handle's lifetime; a bf16 handle's GEMMs read the
 *     projection matrices from the caller's tile-packed copy that
 *     pe_pack_weights fills, so later writes to the row-major matrices are not
 *     seen until they are packed again).  Layouts are dense row-major.  No
 *     call allocates device memory.
 *   - Floating tensors have the handle's dtype: float (PE_DTYPE_F32) or bf16
 *     bit patterns (PE_DTYPE_BF16), except where a signature says float.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on it: no allocation, no host
 *     synchronisation (pe_read_status excepted), no stream creation, so a step
 *     can be captured in a CUDA graph.  Host-side sizes (B, T_in, ...) are
 *     baked into a capture.
 *   - `ws` is a caller-allocated device workspace of at least
 *     pe_workspace_bytes() bytes, 256-byte aligned.  One workspace must not be
 *     used by two calls that may run concurrently.
 *   - Kernels are launched with programmatic stream serialisation: each one may
 *     start its independent prologue (and pull its weights into L2) while the
 *     previous kernel on the stream finishes, and waits for it before reading
 *     its results.
 *   - Return value: PE_OK, or an error code below.  PE_ERR_ARG / PE_ERR_UNSUPPORTED
 *     are detected on the host before anything is enqueued.  PE_ERR_CUDA means
 *     a launch failed (cudaGetLastError).  Problems that only the device can see
 *     (an out-of-range accepted count, block id or token id, an exhausted bounded
 *     wait) do not fault: the kernel clamps or skips the access and ORs a bit
 *     into the status word in `ws`; read it with pe_read_status after the work.
 *   - No exception crosses this interface.
 */
#ifndef PE_H
#define PE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define PE_OK 0
#define PE_ERR_ARG 1          /* null pointer, bad size, workspace too small */
#define PE_ERR_UNSUPPORTED 2  /* dims outside what the kernels handle */
#define PE_ERR_CUDA 3         /* a CUDA runtime call or launch failed */
#define PE_ERR_DEVICE_INPUT 4 /* pe_read_status: the status word has input bits */
#define PE_ERR_TIMEOUT 5      /* pe_read_status: a bounded device wait gave up */

/* device status word bits (pe_read_status) */
#define PE_ST_ACCEPTED_RANGE 0x1u /* a_r outside [0, n_r-1] (clamped) or n_r < 1 */
#define PE_ST_BLOCK_RANGE 0x2u    /* position past the block table, block id outside
                                     [0, num_blocks) or negative position: slot -1,
                                     the key is skipped by attention */
#define PE_ST_TOKEN_RANGE 0x4u    /* token id outside [0, V): embedding row 0 is used */
#define PE_ST_ROWS_RANGE 0x8u     /* pe_verify_greedy: qsl is not a non-decreasing run
                                     from 0 to T_in (each request is clamped to
                                     the rows in range); pe_draft_step with
                                     several layers: a request has more
                                     non-rejected rows than the layers carry */
#define PE_ST_TIMEOUT 0x10u       /* a bounded wait inside a kernel expired */
#define PE_ST_CAPACITY 0x20u      /* COD calls: a sequence length outside [0, S_max]
                                     (clamped), a mask larger than its row capacity
                                     or row stride (rows / columns past it are not
                                     written), or index lists the mask call cannot
                                     have been given by pe_cod_sample_indices
                                     (those rows are skipped) */

/* padding slot of rejected rows ("KV cache and CUDA graphs") */
#define PE_PADDING_SLOT_ID (-1)

enum { PE_DTYPE_F32 = 0, PE_DTYPE_BF16 = 1 };

/* Drafter and step dimensions.  Supported: n_streams == 3; d, inter and
 * head_dim multiples of 8 (16-byte rows); n_heads a multiple of n_kv_heads;
 * head_dim <= 128 (bf16 needs 64 or 128); 1 <= K <= 64; block_size >= 1;
 * K * n_heads / n_kv_heads <= 128 for bf16. */
typedef struct pe_dims {
  int32_t d;          /* drafter hidden size (and each captured stream's width) */
  int32_t n_streams;  /* captured target streams: h_low, h_mid, h_high (3) */
  int32_t n_heads;    /* H, query heads */
  int32_t n_kv_heads; /* G, KV heads; query head h reads KV head h / (H/G) */
  int32_t head_dim;   /* hd */
  int32_t inter;      /* I, SwiGLU intermediate size */
  int32_t vocab;      /* V */
  int32_t K;          /* draft depth: K draft tokens per request */
  int32_t block_size; /* bs, tokens per paged-KV block */
  int32_t mask_id;    /* MASK token id written into the parallel-draft slots */
  int32_t post_norm;  /* 0: pre-norm layer; 1: post-norm layer */
  int32_t dtype;      /* PE_DTYPE_F32 or PE_DTYPE_BF16 */
  float eps;          /* RMSNorm epsilon */
  float rope_theta;   /* RoPE base */
  int32_t n_layers;   /* N decoder layers, 1..PE_MAX_LAYERS (0 is read as 1) */
} pe_dims;

/* Most decoder layers a handle takes. */
#define PE_MAX_LAYERS 16

/* Parameters of decoder layers 2..N (device pointers, borrowed like pe_weights;
 * the same shapes and meanings as the layer fields of pe_weights, which hold
 * layer 1).  gamma_final: post-norm, the norm after this layer's MLP residual;
 * pre-norm, only the last layer's is used, as the final norm. */
typedef struct pe_layer_weights {
  const void* gamma_in;     /* [d] pre-norm only */
  const void* w_qkv;        /* [(H+2G)*hd][d] */
  const void* w_o;          /* [d][H*hd] */
  const void* gamma_post;   /* [d] */
  const void* w_gate;       /* [I][d] */
  const void* w_up;         /* [I][d] */
  const void* w_down;       /* [d][I] */
  const void* gamma_final;  /* [d] */
  const void* attn_sink;    /* [H] float, nullable */
} pe_layer_weights;

/* Drafter parameters: device pointers, borrowed for the handle's lifetime.
 * emb, emb_mask, h_shared and gamma_stream are required.  The layer's parameters
 * (w_fc, w_qkv, w_o, gamma_post, w_gate, w_up, w_down, gamma_final, w_lm, and
 * gamma_in for a pre-norm layer) come all together or all NULL: with none, the
 * handle serves pe_prepare_inputs only and the layer's calls (pe_draft_step,
 * pe_argmax, pe_argmax_noalloc) return PE_ERR_ARG.  Some but not all: PE_ERR_ARG.
 * attn_sink is optional either way. */
typedef struct pe_weights {
  const void* emb;          /* [V][d] token embedding */
  const void* emb_mask;     /* [d] learned emb(mask) for the MASK slots */
  const void* h_shared;     /* [d] learned shared hidden state for the MASK slots,
                               placed in all three stream slots */
  const void* gamma_stream; /* [3][d] RMSNorm gains of the captured streams */
  const void* w_fc;         /* [d][4d] fc: [h_low | h_mid | h_high | emb] -> d */
  const void* gamma_in;     /* [d] pre-norm: norm before QKV (unused post-norm) */
  const void* w_qkv;        /* [(H+2G)*hd][d]: H q heads, then G k, then G v heads */
  const void* w_o;          /* [d][H*hd] */
  const void* gamma_post;   /* [d] pre-norm: MLP input norm; post-norm: norm after
                               the attention residual */
  const void* w_gate;       /* [I][d] */
  const void* w_up;         /* [I][d] */
  const void* w_down;       /* [d][I] */
  const void* gamma_final;  /* [d] pre-norm: final norm; post-norm: norm after the
                               MLP residual */
  const void* w_lm;         /* [V][d] LM head */
  const void* attn_sink;    /* [H] float (in both dtypes), nullable: per-head sink
                               logit of the GPT-oss attention ("Attention Drift",
                               section 3: a learned bias logit in each head's
                               softmax denominator).  It joins the softmax as one
                               more logit with a zero value row.  NULL: no sink */
  const pe_layer_weights* more_layers; /* HOST array of n_layers - 1 entries (layers
                               2..N; read by pe_create only), NULL for one layer */
  const void* packed;       /* bf16 handles with a layer: the tile-packed copy of the
                               projection matrices (pe_pack_weights), caller-owned,
                               256-byte aligned, borrowed for the handle's lifetime;
                               unused (may be NULL) in fp32 mode */
  size_t packed_bytes;      /* its size, at least pe_packed_weights_bytes(dims) */
} pe_weights;

/* Drafter-batch metadata: caller-owned device buffers written by
 * pe_prepare_inputs and read by pe_draft_step.  T_out = T_in + B*(K-1).
 * Request r's output rows are out_qsl[r] .. out_qsl[r+1]-1: its n_r copied rows
 * (row j pairs the hidden state of input row j with the next token, the bonus
 * token at j = a_r; rows past a_r are rejected) followed by K-1 MASK rows at
 * positions prev_pos[a_r] + 1 .. + K-1. */
typedef struct pe_meta {
  int32_t* out_qsl;     /* [B+1] output row offsets */
  int32_t* tok;         /* [T_out] drafter input token */
  int64_t* pos;         /* [T_out] position */
  uint8_t* is_rejected; /* [T_out] 1 for rejected rows */
  uint8_t* is_masked;   /* [T_out] 1 for MASK rows */
  int32_t* hidden_src;  /* [T_out] input row of the hidden state, -1 = h_shared */
  int64_t* slot;        /* [T_out] KV slot, PE_PADDING_SLOT_ID for rejected rows */
  int32_t* valid_qsl;   /* [B+1] exclusive scan of a_r + K */
  int32_t* valid_rows;  /* [T_out] output rows that are not rejected, in order;
                           -1 past n_valid */
  int32_t* n_valid;     /* [1] number of non-rejected rows */
  int32_t* sample_idx;  /* [B*K] output row predicting draft k of request r (r*K+k) */
  int32_t* seq_len;     /* [B] cache positions visible after the step: prev_pos[a_r]+K */
} pe_meta;

typedef struct pe_handle pe_handle;

/* Bytes of the tile-packed copy of a bf16 drafter's projection matrices: w_fc,
 * w_qkv, w_o, w_gate, w_up, w_down and w_lm, then w_qkv, w_o, w_gate, w_up and
 * w_down of each later layer, one after another, each starting 256-byte
 * aligned; a matrix [M][K] is stored in blocks of 128 rows x 64 columns, each
 * one contiguous 16 KB run, blocks ordered by column within a row of blocks,
 * zero-padded to whole blocks.  0 for fp32 dims (the fp32 kernels read the
 * row-major matrices) or dims pe_create would refuse. */
size_t pe_packed_weights_bytes(const pe_dims* dims);

/* Fill `packed` (device, caller-owned, packed_bytes >= pe_packed_weights_bytes,
 * 256-byte aligned) with the tile-packed copy of w's projection matrices
 * (w_fc, w_qkv, w_o, w_gate, w_up, w_down, w_lm and more_layers' five; the
 * other fields are not read).  Asynchronous on `stream`: the copy must be
 * complete before a handle over it runs (same stream, or synchronise).  Packing
 * again after the caller changes its matrices updates every handle that
 * borrows the buffer.  PE_ERR_UNSUPPORTED for fp32 or unsupported dims;
 * PE_ERR_ARG for null or misaligned pointers or a buffer too small. */
int pe_pack_weights(const pe_dims* dims, const pe_weights* w, void* packed, size_t packed_bytes,
                    void* stream);

/* Create a handle for one drafter.  Validates dims (PE_ERR_UNSUPPORTED) and
 * pointers (PE_ERR_ARG: a bf16 handle with a layer also needs w->packed, filled
 * by pe_pack_weights), selects the kernels and encodes the TMA descriptors of
 * the packed weight matrices.  Allocates no device memory and does not
 * synchronise; the handle is a host object.  Uses the current CUDA device;
 * *out is NULL on error. */
int pe_create(const pe_dims* dims, const pe_weights* w, pe_handle** out);

/* Destroy a handle (NULL is ignored).  It never frees the caller's weights or
 * packed copy.  No work that uses the handle may still be in flight. */
void pe_destroy(pe_handle* h);

/* Workspace bytes that cover every call with at most max_batch requests,
 * max_rows_in previous verify rows in total and block tables of at most
 * max_blocks_per_seq entries per request.  0 on bad arguments. */
size_t pe_workspace_bytes(const pe_handle* h, int max_batch, int max_rows_in,
                          int max_blocks_per_seq);

/* Steps (1)-(3): batch metadata, hidden-state map and drafter input.
 *   qsl[B+1]        int32, input row offsets of the previous verify batch
 *   prev_tok[T_in]  int32 token ids;  prev_pos[T_in] int64 positions
 *   accepted[B]     int32 a_r, accepted drafts, 0 <= a_r <= n_r - 1
 *   bonus[B]        int32 bonus (correction) token b_r
 *   block_table[B][max_blocks] int32 physical KV block ids; num_blocks bounds them
 *   H_tgt[T_in][3][d] captured target hidden states (h_low, h_mid, h_high)
 *   meta            output metadata buffers (all fields required)
 *   G_out  [T_out][3][d]  nullable: hidden-state map; MASK rows get h_shared
 *   E_out  [T_out][d]     nullable: embedding rows; MASK rows get emb(mask)
 *   A_out  [T_out][4d]    nullable: drafter input of the non-rejected rows in
 *                         valid_rows order (row i <-> valid_rows[i]):
 *                         [RMSNorm(h_low), RMSNorm(h_mid), RMSNorm(h_high), emb]
 * Clears the status word in ws, then ORs in any input problem it finds. */
int pe_prepare_inputs(pe_handle* h, int B, int T_in, const int32_t* qsl,
                      const int32_t* prev_tok, const int64_t* prev_pos,
                      const int32_t* accepted, const int32_t* bonus,
                      const int32_t* block_table, int max_blocks, int num_blocks,
                      const void* H_tgt, const pe_meta* meta, void* G_out, void* E_out,
                      void* A_out, void* ws, size_t ws_bytes, void* stream);

/* Step (4): the drafter layer for the batch prepared by pe_prepare_inputs.
 *   A         [T_out][4d] drafter input from pe_prepare_inputs (A_out)
 *   k_cache, v_cache  [n_layers][num_blocks][G][block_size][hd] paged KV
 *             caches, one per layer, back to back; this step's non-rejected rows
 *             are written at meta->slot (never at -1) in every layer, then
 *             attention reads them back
 * With n_layers > 1 every layer but the last runs over all non-rejected rows
 * ("Parallel drafting": all positions pass through the N layers), laid out per
 * request in R = min(2K, 128 / (H/G)) rows (2K in fp32 mode), right-aligned.  A
 * request whose a_r + K non-rejected rows exceed R (a prefill-sized request)
 * sets PE_ST_ROWS_RANGE and its drafts are not valid; steady-state steps
 * (n_r <= K + 1 verify rows) always fit.
 *   z_out     [B*K][d] normalised final hidden state of the K sample rows of each
 *             request (row r*K + k predicts draft token k+1 of request r)
 * block_table / max_blocks / num_blocks as passed to pe_prepare_inputs. */
int pe_draft_step(pe_handle* h, int B, int T_in, const pe_meta* meta, const void* A,
                  const int32_t* block_table, int max_blocks, int num_blocks,
                  void* k_cache, void* v_cache, void* z_out, void* ws, size_t ws_bytes,
                  void* stream);

/* Step (5): LM head fused with argmax.  draft_tokens[n] = argmax_v z[n] . w_lm[v]
 * (lowest index on ties; fp32 logits).  logits [n_rows][V] float is nullable:
 * when given, the fp32 logits are stored too. */
int pe_argmax(pe_handle* h, const void* z, int n_rows, int32_t* draft_tokens, float* logits,
              void* ws, size_t ws_bytes, void* stream);

/* The autoregressive drafting that the parallel step replaces, on the same
 * kernels: K sequential passes of the one-layer drafter, one draft token per
 * pass ("P-EAGLE: parallel speculative decoding in vLLM", Solving the
 * autoregressive drafting bottleneck: K drafts cost K sequential forward
 * passes; "Attention Drift", sections 3 and 4.1: after the first step the
 * drafter consumes its own hidden state).
 *   pass 1      the parallel step with one draft row per request: metadata,
 *               drafter input, layer and LM head over the non-rejected rows of
 *               the verify batch, the NTP row (bonus token, target hidden state)
 *               drafting token 1;
 *   pass k > 1  one row per request at position prev_pos[a_r] + k - 1 (where
 *               the parallel step puts MASK row k - 1), its three stream slots
 *               filled with the drafter's own hidden state of pass k - 1 (y of a
 *               pre-norm layer, the normalised output of a post-norm layer, both
 *               fp32) and its token slot with the embedding of draft k - 1.
 * Every pass writes its rows' KV (k_cache, v_cache as for pe_draft_step, the
 * slots of the parallel step's non-rejected rows) and attends to the cache
 * after its own write.
 * Inputs as for pe_prepare_inputs (no metadata buffers: they live in ws).
 *   draft_tokens [B][K] int32 out: draft k of request r at r * K + k - 1
 *   logits       [B][K][V] float, nullable: each pass's fp32 logits
 *   hidden_out   [B][K][d] float, nullable: the hidden state each pass hands
 *                to the next (the drafter output "Attention Drift" Table 1
 *                tracks per speculative step)
 *   ws           pe_autoregressive_workspace_bytes(...) bytes or more, 256-byte
 *                aligned; its status word is cleared first (pe_read_status)
 * One decoder layer only: a handle with n_layers > 1 returns
 * PE_ERR_UNSUPPORTED.  PE_ERR_ARG as for pe_prepare_inputs / pe_draft_step.
 * All K passes are enqueued on `stream` (3 + 14 K kernels in bf16 mode); no host
 * round trip between passes: each pass reads the previous pass's draft and
 * hidden state on the device. */
size_t pe_autoregressive_workspace_bytes(const pe_handle* h, int max_batch, int max_rows_in,
                                         int max_blocks_per_seq);
int pe_draft_autoregressive(pe_handle* h, int B, int T_in, const int32_t* qsl,
                            const int32_t* prev_tok, const int64_t* prev_pos,
                            const int32_t* accepted, const int32_t* bonus,
                            const int32_t* block_table, int max_blocks, int num_blocks,
                            const void* H_tgt, void* k_cache, void* v_cache, int32_t* draft_tokens,
                            float* logits, float* hidden_out, void* ws, size_t ws_bytes,
                            void* stream);

/* Allocation-free pe_argmax.  The pages have no counterpart: this is an
 * interface addition for callers that cannot allocate device memory at all,
 * such as a serving engine that has already reserved every byte for weights and
 * KV cache and hands a plugin only a stream, or a runtime bound to a fixed
 * memory plan.
 * Same arguments and results as pe_argmax, without the workspace: its scratch
 * (one 64-bit argmax key per row) lives in a static device array of
 * PE_NOALLOC_MAX_ROWS entries (32 KiB) that every GPU loading this library holds
 * until the process exits.  n_rows above PE_NOALLOC_MAX_ROWS returns PE_ERR_ARG.
 * The call performs no cudaMalloc / cudaFree and runs pe_argmax's LM-head plan
 * (its K splits add their partial tiles inside a thread-block cluster, with no
 * global scratch).  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current and caches it for the
 * process (one context per device: do not call it again on a device after a
 * cudaDeviceReset); make that first call before any stream capture.  All calls
 * on a device share the array: each call clears the keys it uses, and calls
 * that overlap on the GPU race.  No status word is kept, so device-side problems
 * are not reported. */
#define PE_NOALLOC_MAX_ROWS 4096
int pe_argmax_noalloc(pe_handle* h, const void* z, int n_rows, int32_t* draft_tokens,
                      float* logits, void* stream);

/* Greedy verification of the drafts: the step that produces the next
 * pe_prepare_inputs' accepted counts and bonus tokens.  "Attention Drift",
 * section 2 (preliminaries): the target scores the drafted tokens in one forward
 * pass and keeps the longest prefix it accepts; with greedy drafts that is
 * exact agreement with the target's greedy token.  Needs no handle.
 *   qsl[B+1]       int32 row offsets of the verify batch: request r owns rows
 *                  qsl[r] .. qsl[r+1]-1 (n_r >= 0 rows); qsl[0] = 0, qsl[B] = T_in
 *   tok[T_in]      int32 token of each verify row: row 0 of a request holds the
 *                  last committed token, row j >= 1 its draft j
 *   logits         [T_in][vocab] the target's logits after each row's token,
 *                  float (PE_DTYPE_F32) or bf16 bits (PE_DTYPE_BF16); rows need
 *                  no particular alignment beyond the element size
 *   target_tok[T_in] out: greedy token of each row (largest logit, lowest index
 *                  on ties, -0 equal to +0, a NaN above every number)
 *   accepted[B]    out: a_r = the largest m <= n_r - 1 with tok[qsl[r]+j] ==
 *                  target_tok[qsl[r]+j-1] for every j = 1..m
 *   bonus[B]       out: target_tok[qsl[r] + a_r] (the correction or next token);
 *                  a request with no rows gets accepted 0 and bonus -1
 *   ws             device workspace of pe_verify_workspace_bytes(T_in, vocab)
 *                  bytes or more, 256-byte aligned; its first word is the status
 *                  word (read with pe_read_status, handle NULL allowed)
 * The logits are read once (the call is bound by their bytes).  A qsl that is
 * not a non-decreasing run from 0 to T_in sets PE_ST_ROWS_RANGE and each request
 * is clamped to the rows in range; rows outside every request get no target
 * token.  PE_ERR_ARG: negative sizes, null pointers, logits not aligned to the
 * element size, ws misaligned or too small, B = 0 with T_in > 0. */
size_t pe_verify_workspace_bytes(int max_rows_in, int vocab);
int pe_verify_greedy(int B, int T_in, const int32_t* qsl, const int32_t* tok,
                     const void* logits, int vocab, int dtype, int32_t* target_tok,
                     int32_t* accepted, int32_t* bonus, void* ws, size_t ws_bytes,
                     void* stream);

/* ---------------------------------------------------------------- COD training indices
 * "[RFC]: Add random anchor for p-eagle first position": the training-side
 * index lists of COD sampling and the asymmetric attention mask built on them.
 * For a batch of B sequences (sequence b has seq_len[b] <= S_max tokens; every
 * per-sequence array has row stride S_max):
 *   depth 0 (anchors)  the positions with loss_mask != 0; when max_anchors > 0
 *                      and there are more of them, the max_anchors with the
 *                      smallest (u_anchor, position) keys, i.e. a uniform random
 *                      subset for uniform draws
 *   depth k (1..D-1)   the anchors of depth k-1 with u_keep[k-1][a] < retain
 *                      and a + k < seq_len (each chain continues on its own
 *                      draw; the page's "drop rate" is this retained share)
 * Query rows of the mask: the COD tokens, depth-major (depth 0's anchors, then
 * depth 1's, ...), anchors ascending within a depth; row (a, k) stands at
 * position a + k.  Key columns: the seq_len original positions, then the depth
 * >= 1 tokens in the same order.  Row (a, k) may attend original position j iff
 * j <= a, and chain token (a', k') iff a' == a and k' <= k (the reply's "Depth >
 * 0 attention": the original sequence up to the anchor plus its own chain).
 * Sizes: Q = sum_k counts[k] rows, KV = seq_len + Q - counts[0] columns.
 *
 * The random draws are inputs: float in [0, 1) (negative or NaN draws are
 * outside the contract).  Both calls are asynchronous on `stream` and capturable. */
#define PE_COD_MAX_DEPTH 16

/* Workspace for both COD calls: 256 + B * (n_depth - 1) * S_max * 4 bytes (the
 * status word, then each chain member's place in its depth's list, which
 * pe_cod_sample_indices writes and pe_cod_mask reads).  0 for invalid sizes. */
size_t pe_cod_workspace_bytes(int B, int S_max, int n_depth);

/* COD index lists.
 *   seq_len[B]            int32 sequence lengths (outside [0, S_max]: clamped,
 *                         PE_ST_CAPACITY)
 *   loss_mask[B][S_max]   uint8, non-zero = the position carries a loss
 *   n_depth               D, 1..PE_COD_MAX_DEPTH
 *   retain                share of a depth's chains kept for the next depth
 *   max_anchors           cap on depth-0 anchors per sequence, 0 = no cap
 *   u_anchor[B][S_max]    float draws of the anchor subset
 *   u_keep[B][D-1][S_max] float draws of the chain continuations (NULL if D = 1)
 *   idx[B][D][S_max]      out: idx[b][k][0..counts[b][k]) = depth k's anchor
 *                         positions, ascending; the rest of each row is not written
 *   counts[B][D]          out: list lengths
 *   ws                    pe_cod_workspace_bytes(B, S_max, D) bytes or more,
 *                         256-byte aligned; the call clears its status word
 * PE_ERR_ARG: negative sizes, D outside 1..16, NaN retain, negative cap, null
 * or misaligned pointers, ws too small.  PE_ERR_UNSUPPORTED: B > 65535. */
int pe_cod_sample_indices(int B, int S_max, const int32_t* seq_len, const uint8_t* loss_mask,
                          int n_depth, float retain, int max_anchors, const float* u_anchor,
                          const float* u_keep, int32_t* idx, int32_t* counts, void* ws,
                          size_t ws_bytes, void* stream);

/* The asymmetric mask of each sequence, from the lists of pe_cod_sample_indices
 * (same B, S_max, seq_len, D and ws).
 *   mask                  uint8, sequence b's mask at mask + b * mask_stride:
 *                         row q at + q * ld, 1 = may attend, 0 = masked.  Rows
 *                         0..Q-1 are written, each up to the next multiple of 16
 *                         bytes past its KV columns (the extra bytes 0); rows >= Q
 *                         and columns beyond are left untouched.
 *   q_cap                 rows each sequence's block holds (>= Q; D * the anchor
 *                         count is always enough)
 *   ld                    row stride in bytes, a multiple of 16, >= KV rounded up
 *                         to 16 (S_max + (D-1) * anchors is always enough)
 *   mask_stride           bytes between sequences, a multiple of 16, >= q_cap * ld
 * A mask larger than q_cap or ld sets PE_ST_CAPACITY and writes what fits.  The
 * status word is not cleared (read it after both calls).  PE_ERR_ARG: as above,
 * plus a misaligned mask, ld or mask_stride. */
int pe_cod_mask(int B, int S_max, const int32_t* seq_len, int n_depth, const int32_t* idx,
                const int32_t* counts, uint8_t* mask, int64_t q_cap, int64_t ld,
                int64_t mask_stride, void* ws, size_t ws_bytes, void* stream);

/* Copy the device status word from ws into *status (synchronises `stream`);
 * clear it when `clear` is non-zero.  Returns PE_OK when no bit is set,
 * PE_ERR_TIMEOUT when PE_ST_TIMEOUT is set, else PE_ERR_DEVICE_INPUT.  h may be
 * NULL (the word lives in ws; pe_verify_greedy has no handle). */
int pe_read_status(const pe_handle* h, void* ws, uint32_t* status, int clear, void* stream);

/* Static text for a return code. */
const char* pe_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* PE_H */
