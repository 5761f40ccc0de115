// C-ABI of the P-EAGLE parallel-draft step: handle, workspace layout and the
// three step calls (include/pe.h documents every argument).
//
// All work is enqueued on the caller's stream; nothing here allocates device
// memory, synchronises the host or creates streams, except pe_read_status, which
// synchronises the stream to read the status word back.  The tile-packed copy
// of a bf16 drafter's projection weights lives in a caller-owned buffer that
// pe_pack_weights fills and pe_create borrows.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "pe_internal.h"
#include "pe_prep.h"
#include "pe_testing.h"

using namespace pe;

// Decoder layers 2..N: their parameters and the tensor maps of their packed
// projection weights (layer 1's live in pe_weights and the handle's own maps).
struct LayerSlot {
  pe_layer_weights w;
  CUtensorMap m_qkv, m_o, m_gate, m_up, m_down;
};

struct pe_handle {
  pe_dims d;
  pe_weights w;
  int num_sms;
  CUtensorMap m_fc, m_qkv, m_o, m_gate, m_up, m_down, m_lm;
  uint64_t rope_turn[64];  // RoPE frequencies as fractions of a turn (rope_cos_sin)
  bool has_layer;  // false: metadata / drafter-input handle without layer weights
  int n_layers;
  LayerSlot more[PE_MAX_LAYERS - 1];  // layers 2..n_layers
};

namespace {

enum GemmId { G_FC = 0, G_QKV, G_O, G_GATEUP, G_DOWN, G_LM, G_COUNT };

size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Dimensions the kernels handle (PE_OK) or not (PE_ERR_UNSUPPORTED).
int check_dims(const pe_dims& d) {
  if (d.dtype != PE_DTYPE_BF16 && d.dtype != PE_DTYPE_F32) return PE_ERR_UNSUPPORTED;
  if (d.n_streams != 3 || d.d <= 0 || d.d % 8 || d.inter <= 0 || d.inter % 8 || d.vocab <= 0 ||
      d.n_heads <= 0 || d.n_kv_heads <= 0 || d.n_heads % d.n_kv_heads || d.head_dim <= 0 ||
      d.head_dim % 8 || d.head_dim > 128 || d.K < 1 || d.K > 64 || d.block_size < 1 ||
      !(d.eps >= 0.f) || !(d.rope_theta > 0.f) || d.n_layers > PE_MAX_LAYERS)
    return PE_ERR_UNSUPPORTED;
  if (d.dtype == PE_DTYPE_BF16 &&
      ((d.head_dim != 64 && d.head_dim != 128) || d.K * (d.n_heads / d.n_kv_heads) > 128))
    return PE_ERR_UNSUPPORTED;
  return PE_OK;
}

// The projection matrices a bf16 handle reads tile-packed, in their order in
// the caller's packed buffer (each copy starts 256-byte aligned): w_fc, w_qkv,
// w_o, w_gate, w_up, w_down, w_lm, then w_qkv, w_o, w_gate, w_up, w_down of each
// later layer.  w may be NULL (sizes only).
struct PackedMat {
  const void* W;
  int M, K;
  size_t off;
};

std::vector<PackedMat> packed_mats(const pe_dims& d, const pe_weights* w, size_t* total) {
  const int n_layers = d.n_layers <= 0 ? 1 : d.n_layers;
  const int QKV = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
  const int HD = d.n_heads * d.head_dim;
  std::vector<PackedMat> m = {{w ? w->w_fc : nullptr, d.d, 4 * d.d, 0},
                              {w ? w->w_qkv : nullptr, QKV, d.d, 0},
                              {w ? w->w_o : nullptr, d.d, HD, 0},
                              {w ? w->w_gate : nullptr, d.inter, d.d, 0},
                              {w ? w->w_up : nullptr, d.inter, d.d, 0},
                              {w ? w->w_down : nullptr, d.d, d.inter, 0},
                              {w ? w->w_lm : nullptr, d.vocab, d.d, 0}};
  for (int l = 0; l < n_layers - 1; ++l) {
    const pe_layer_weights* lw = w && w->more_layers ? &w->more_layers[l] : nullptr;
    m.push_back({lw ? lw->w_qkv : nullptr, QKV, d.d, 0});
    m.push_back({lw ? lw->w_o : nullptr, d.d, HD, 0});
    m.push_back({lw ? lw->w_gate : nullptr, d.inter, d.d, 0});
    m.push_back({lw ? lw->w_up : nullptr, d.inter, d.d, 0});
    m.push_back({lw ? lw->w_down : nullptr, d.d, d.inter, 0});
  }
  size_t off = 0;
  for (auto& x : m) {
    x.off = off;
    off += al256(packed_weight_bytes(x.M, x.K));
  }
  *total = off;
  return m;
}
size_t esize(const pe_handle* h) { return h->d.dtype == PE_DTYPE_BF16 ? 2 : 4; }
bool is_bf16(const pe_handle* h) { return h->d.dtype == PE_DTYPE_BF16; }

struct GemmShape {
  int M, K, dual;
};

GemmShape gemm_shape(const pe_handle* h, int id) {
  const pe_dims& d = h->d;
  switch (id) {
    case G_FC: return {d.d, 4 * d.d, 0};
    case G_QKV: return {(d.n_heads + 2 * d.n_kv_heads) * d.head_dim, d.d, 0};
    case G_O: return {d.d, d.n_heads * d.head_dim, 0};
    case G_GATEUP: return {d.inter, d.d, 1};
    case G_DOWN: return {d.d, d.inter, 0};
    default: return {d.vocab, d.d, 0};
  }
}

TcPlan plan_of(const pe_handle* h, int id, int N, bool bpair, bool allow_split = true,
               bool partial = false) {
  const GemmShape s = gemm_shape(h, id);
  return plan_gemm_tc(s.M, s.K, N, s.dual, bpair ? 1 : 0, h->num_sms, allow_split, partial);
}

// The projections whose K splits store partial sums (EPI_PARTIAL_F32) for the
// kernel after them to add, and whether their token operand is a bf16 pair.
bool partial_gemm(int id) { return id == G_FC || id == G_QKV || id == G_O || id == G_DOWN; }
bool pair_operand(int id) { return id == G_QKV || id == G_GATEUP || id == G_DOWN; }

// Bytes of partial sums projection `id` stores over any N <= N_max token rows
// (the split count rises as N falls, so every N is walked).
size_t partial_bytes_bound(const pe_handle* h, int id, int N_max) {
  const GemmShape s = gemm_shape(h, id);
  if (!is_bf16(h) || !partial_gemm(id)) return static_cast<size_t>(N_max) * s.M * sizeof(float);
  size_t best = 0;
  for (int n = 1; n <= N_max; ++n) {
    const TcPlan p = plan_of(h, id, n, pair_operand(id), true, true);
    best = std::max(best, static_cast<size_t>(p.partial ? p.k_splits : 1) * n * s.M * sizeof(float));
  }
  return best;
}

// Rows per request that the attention, O and MLP steps carry: the K sample rows
// with one layer; with several, every non-rejected row (a_r + K <= 2K for n_r <=
// K + 1), right-aligned, as many as one attention tile of the bf16 kernel holds.
int layer_rows(const pe_handle* h) {
  const pe_dims& d = h->d;
  if (h->n_layers <= 1) return d.K;
  int R = 2 * d.K;
  if (is_bf16(h)) R = std::min(R, 128 / (d.n_heads / d.n_kv_heads));
  return R;
}

// Attention split partials, bounded over every batch size <= B (the split count
// rises as the batch shrinks).
size_t attn_scratch_bound(const pe_handle* h, int B, int max_blocks, int rows) {
  if (!is_bf16(h)) return 0;
  const pe_dims& d = h->d;
  size_t best = 0;
  // the split count only grows with the block-table width, so the width given
  // bounds every narrower call; the batch size is walked
  for (int b = 1; b <= B; ++b) {
    const int ns = attention_split_count(b, d.n_kv_heads, max_blocks, d.block_size, h->num_sms);
    best = std::max(best, attention_scratch_bytes(b, rows, d.n_heads, d.head_dim, ns));
  }
  return best;
}

struct Layout {
  // x: fc output (fp32); u / u_lo: QKV operand (bf16 pair; fp32 in fp32 mode);
  // q_s; x_s: residual rows (fp32); attn; r: attention residual sum (fp32);
  // a / a_lo / a_f: MLP operand pair and its fp32 value; h / h_lo: SwiGLU
  // product pair; part: the split partial sums of fc, QKV, O and down (one at
  // a time: each is read by the next kernel before the next projection stores);
  // amax: argmax keys; tok: the test hook's argmax indices
  size_t status, x, u, u_lo, q_s, x_s, attn, r, a, a_lo, a_f, h, h_lo, part, amax, attn_part, tok;
  // several layers: a later layer's input, fp32 (xl) and as its QKV operand (ul, ul_lo)
  size_t xl, ul, ul_lo;
  size_t dec;  // persistent decode layer: partial tiles and operands
  size_t total;
};

// Barrier words of the persistent decode layer: in the workspace header, after
// the status word (the header's 256 bytes are cleared together).
constexpr size_t kBarrierWordsOffset = 64;
// the first kernel's launch count is barrier word 12 (pe_decode.cu)
static_assert(kBarrierWordsOffset + 4 * 12 == PE_TEST_DECODE_EPOCH_BYTE, "decode epoch word");

// Workspace layout of a step with B requests, T_in verify rows and block tables
// of max_blocks entries.  Each region is sized by a bound that only grows with
// (B, T_in, max_blocks), so a workspace sized for the maxima fits every call.
// K_draft: draft rows per request of the step (0: the handle's K; the
// autoregressive passes run single-draft steps).
Layout layout_of(const pe_handle* h, int B, int T_in, int max_blocks, int K_draft = 0) {
  const pe_dims& d = h->d;
  const size_t e = esize(h);
  const int Kd = K_draft > 0 ? K_draft : d.K;
  const int rows = K_draft > 0 ? K_draft : layer_rows(h);
  const int T_out = T_in + B * (Kd - 1);
  const int NS = B * rows;
  const int Hd = d.n_heads * d.head_dim;
  const int QKV = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
  const bool layers = h->n_layers > 1;
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = al256(off + bytes);
    return o;
  };
  L.status = take(256);
  const size_t f4 = sizeof(float);
  L.x = take(static_cast<size_t>(T_out) * d.d * f4);
  L.u = take(static_cast<size_t>(T_out) * d.d * f4);
  L.u_lo = take(static_cast<size_t>(T_out) * d.d * e);
  L.q_s = take(static_cast<size_t>(NS) * Hd * e);
  L.x_s = take(static_cast<size_t>(NS) * d.d * f4);
  L.attn = take(static_cast<size_t>(NS) * Hd * e);
  L.r = take(static_cast<size_t>(NS) * d.d * f4);
  L.a = take(static_cast<size_t>(NS) * d.d * f4);
  L.a_lo = take(static_cast<size_t>(NS) * d.d * e);
  L.a_f = take(static_cast<size_t>(NS) * d.d * f4);
  L.h = take(static_cast<size_t>(NS) * d.inter * f4);
  L.h_lo = take(static_cast<size_t>(NS) * d.inter * e);
  L.part = take(std::max(std::max(partial_bytes_bound(h, G_FC, T_out),
                                  partial_bytes_bound(h, G_QKV, layers ? std::max(T_out, NS) : T_out)),
                         std::max(partial_bytes_bound(h, G_O, NS),
                                  partial_bytes_bound(h, G_DOWN, NS))));
  if (layers) {
    L.xl = take(static_cast<size_t>(NS) * d.d * f4);
    L.ul = take(static_cast<size_t>(NS) * d.d * f4);
    L.ul_lo = take(static_cast<size_t>(NS) * d.d * e);
  }
  L.amax = take(static_cast<size_t>(NS) * sizeof(unsigned long long));
  L.attn_part = take(attn_scratch_bound(h, B, max_blocks, rows));
  if (is_bf16(h) && h->n_layers <= 1 && decode_layer_fits(d.d, QKV, d.inter, h->num_sms))
    L.dec = take(decode_scratch_bytes(d.d, QKV, d.inter, h->num_sms));
  L.total = off;
  return L;
}

// Workspace of pe_argmax for n_rows rows.
Layout layout_argmax(const pe_handle* h, int n_rows) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = al256(off + bytes);
    return o;
  };
  L.status = take(256);
  L.amax = take(static_cast<size_t>(n_rows) * sizeof(unsigned long long));
  L.total = off;
  return L;
}

// Workspace of one projection (test hook) over n_rows rows.
// The test hook's workspace: the status word; with the argmax epilogue, the
// row keys and the row maxima's indices (at PE_PROJ_ARGMAX_TOKENS_OFFSET).
Layout layout_projection(const pe_handle* h, int which, int n_rows, bool argmax = false) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = al256(off + bytes);
    return o;
  };
  L.status = take(256);
  if (argmax) {
    L.amax = take(static_cast<size_t>(n_rows) * sizeof(unsigned long long));
    L.tok = take(static_cast<size_t>(n_rows) * sizeof(int32_t));
  }
  (void)h;
  (void)which;
  L.total = off;
  return L;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

int check_meta(const pe_meta* m) {
  if (!m || !m->out_qsl || !m->tok || !m->pos || !m->is_rejected || !m->is_masked ||
      !m->hidden_src || !m->slot || !m->valid_qsl || !m->valid_rows || !m->n_valid ||
      !m->sample_idx || !m->seq_len)
    return PE_ERR_ARG;
  return PE_OK;
}

// One projection of the step, on the tensor cores (bf16) or SIMT (fp32).
// X_lo: the low half of a bf16-pair operand (bf16 only; nullable).
// epi.mode EPI_PARTIAL_F32: *n_parts receives the number of partial tiles stored.
int run_gemm(pe_handle* h, int id, const void* X, const void* X_lo, int N_cap,
             const int* n_rows_dev, const Epilogue& epi, void* ws, const Layout& L,
             cudaStream_t st, bool allow_split = true, int* n_parts = nullptr, int layer = 0) {
  const GemmShape s = gemm_shape(h, id);
  const bool partial = epi.mode == EPI_PARTIAL_F32;
  if (n_parts) *n_parts = 1;
  // layers 2..N: their own projection weights (fc and the LM head are shared)
  const LayerSlot* ls = layer > 0 && id != G_FC && id != G_LM ? &h->more[layer - 1] : nullptr;
  if (!is_bf16(h)) {
    const pe_weights& w = h->w;
    const void* W = id == G_FC ? w.w_fc : id == G_QKV ? (ls ? ls->w.w_qkv : w.w_qkv)
                  : id == G_O ? (ls ? ls->w.w_o : w.w_o)
                  : id == G_GATEUP ? (ls ? ls->w.w_gate : w.w_gate)
                  : id == G_DOWN ? (ls ? ls->w.w_down : w.w_down) : w.w_lm;
    const void* W2 = id == G_GATEUP ? (ls ? ls->w.w_up : w.w_up) : nullptr;
    return launch_gemm_f32(static_cast<const float*>(W), static_cast<const float*>(W2),
                           static_cast<const float*>(X), s.M, s.K, N_cap, n_rows_dev, epi, st);
  }
  const TcPlan p = plan_of(h, id, N_cap, X_lo != nullptr, allow_split, partial);
  if (n_parts) *n_parts = p.partial ? p.k_splits : 1;
  Epilogue ep = epi;
  if (partial && !p.partial) ep.mode = EPI_STORE_F32;  // the splits reduce in a cluster
  const CUtensorMap* mA = id == G_FC ? &h->m_fc : id == G_QKV ? (ls ? &ls->m_qkv : &h->m_qkv)
                        : id == G_O ? (ls ? &ls->m_o : &h->m_o)
                        : id == G_GATEUP ? (ls ? &ls->m_gate : &h->m_gate)
                        : id == G_DOWN ? (ls ? &ls->m_down : &h->m_down) : &h->m_lm;
  const CUtensorMap* mA2 = id == G_GATEUP ? (ls ? &ls->m_up : &h->m_up) : nullptr;
  return launch_gemm_tc(p, mA, mA2, X, X_lo, n_rows_dev, ep, at<uint32_t>(ws, L.status), st);
}

// Device buffers of one step inside the workspace, and the stream.
struct StepCtx {
  pe_handle* h;
  const Layout* L;
  void* ws;
  cudaStream_t st;
  int dt;
  bool bf;
  uint32_t* status;
  float* x;
  void* u;
  bf16_t* u_lo;
  float* part;
  void* q_s;
  float* x_s;
  void* attn;
  float* r;
  void* a;
  bf16_t* a_lo;
  float* a_f;
  void* hm;
  bf16_t* h_lo;
};

StepCtx make_ctx(pe_handle* h, const Layout& L, void* ws, cudaStream_t st) {
  StepCtx c{};
  c.h = h;
  c.L = &L;
  c.ws = ws;
  c.st = st;
  c.dt = h->d.dtype;
  c.bf = c.dt == PE_DTYPE_BF16;
  c.status = at<uint32_t>(ws, L.status);
  c.x = at<float>(ws, L.x);
  c.u = at<void>(ws, L.u);
  c.u_lo = c.bf ? at<bf16_t>(ws, L.u_lo) : nullptr;
  c.part = at<float>(ws, L.part);
  c.q_s = at<void>(ws, L.q_s);
  c.x_s = at<float>(ws, L.x_s);
  c.attn = at<void>(ws, L.attn);
  c.r = at<float>(ws, L.r);
  c.a = at<void>(ws, L.a);
  c.a_lo = c.bf ? at<bf16_t>(ws, L.a_lo) : nullptr;
  c.a_f = at<float>(ws, L.a_f);
  c.hm = at<void>(ws, L.h);
  c.h_lo = c.bf ? at<bf16_t>(ws, L.h_lo) : nullptr;
  return c;
}

// A row norm over the sum of a projection's n_parts partial tiles (plus an
// optional fp32 residual); sum_out (nullable) receives that fp32 sum and
// norm_out (nullable) the normalised value before rounding.
int step_norm(const StepCtx& c, const float* parts, int n_parts, size_t part_stride,
              const float* resid, float* sum_out, const void* gamma, int apply, void* out,
              bf16_t* out_lo, float* out_f32, int rows, const int* n_rows_dev,
              float* norm_out = nullptr) {
  const pe_dims& d = c.h->d;
  RowNormArgs n{};
  n.x = parts;
  n.ld_x = d.d;
  n.n_parts = n_parts;
  n.part_stride = part_stride;
  n.resid = resid;
  n.ld_resid = d.d;
  n.sum_out = sum_out;
  n.norm_out = norm_out;
  n.gamma = gamma;
  n.apply_norm = apply;
  n.out = out;
  n.out_lo = out_lo;
  n.out_f32 = out_f32;
  n.ld_out = d.d;
  n.d = d.d;
  n.eps = d.eps;
  n.rows_cap = rows;
  n.n_rows_dev = n_rows_dev;
  return launch_rownorm(n, c.dt, c.st);
}

// Each projection but gate/up stores the partial sums of its K splits; the
// kernel after it adds them (in split order) as it reads them.
Epilogue partial_epi(const StepCtx& c, int rows, int M) {
  Epilogue ep;
  ep.mode = EPI_PARTIAL_F32;
  ep.out = c.part;
  ep.ld_out = M;
  ep.part_stride = static_cast<size_t>(rows) * M;
  return ep;
}

// fc and its row norm: x = A W_fc^T over the non-rejected rows (fp32, kept for
// the residual) and the QKV operand u = RMSNorm(x; gamma_in) (pre-norm) or x
// (post-norm), a bf16 pair in bf16 mode.
int fc_step(const StepCtx& c, int T_out, const pe_meta* meta, const void* A) {
  pe_handle* h = c.h;
  int np = 1;
  const Epilogue e = partial_epi(c, T_out, h->d.d);
  int rc = run_gemm(h, G_FC, A, nullptr, T_out, meta->n_valid, e, c.ws, *c.L, c.st, true, &np);
  if (rc != PE_OK) return rc;
  return step_norm(c, c.part, np, e.part_stride, nullptr, c.x, h->w.gamma_in,
                   h->d.post_norm ? 0 : 1, c.u, c.u_lo, nullptr, T_out, meta->n_valid);
}

// The attention of the step's sample rows (Kd per request) over the paged cache.
int attention_step(const StepCtx& c, int Kd, int B, const pe_meta* meta, const int32_t* block_table,
                   int max_blocks, int num_blocks, void* k_cache, void* v_cache) {
  pe_handle* h = c.h;
  const pe_dims& d = h->d;
  const int NS = B * Kd;
  AttnArgs aa{};
  aa.B = B;
  aa.K = Kd;
  aa.H = d.n_heads;
  aa.G = d.n_kv_heads;
  aa.hd = d.head_dim;
  aa.bs = d.block_size;
  aa.max_blocks = max_blocks;
  aa.num_blocks = num_blocks;
  plan_attention(B, d.n_kv_heads, Kd, d.n_heads, d.head_dim, max_blocks, d.block_size, h->num_sms,
                 aa.n_splits, aa.split_len, aa.cluster);
  aa.q = c.q_s;
  aa.k_cache = k_cache;
  aa.v_cache = v_cache;
  aa.block_table = block_table;
  aa.seq_len = meta->seq_len;
  aa.part_o = at<float>(c.ws, c.L->attn_part);
  aa.part_ml = reinterpret_cast<float*>(static_cast<char*>(c.ws) + c.L->attn_part +
                                        al256(static_cast<size_t>(aa.n_splits) * NS * d.n_heads *
                                              d.head_dim * sizeof(float)));
  aa.out = c.attn;
  aa.sink = static_cast<const float*>(h->w.attn_sink);
  aa.k_min = Kd;
  aa.status = c.status;
  return launch_attention(aa, c.dt, c.st);
}

// A decode-sized one-layer step (at most 16 token rows and 16 sample rows):
// fc, QKV and RoPE/KV write in one persistent kernel, attention, then O,
// gate/up, down and the final norm in a second (pe_decode.cu).
int decode_layer_step(const StepCtx& c, int Kd, int B, int T_in, const pe_meta* meta,
                      const void* A, const int32_t* block_table, int max_blocks, int num_blocks,
                      void* k_cache, void* v_cache, void* z_out, float* hidden_out) {
  pe_handle* h = c.h;
  const pe_dims& d = h->d;
  DecodeLaunch dl{};
  dl.d = d.d;
  dl.H = d.n_heads;
  dl.G = d.n_kv_heads;
  dl.hd = d.head_dim;
  dl.inter = d.inter;
  dl.K = Kd;
  dl.B = B;
  dl.T_out = T_in + B * (Kd - 1);
  dl.bs = d.block_size;
  dl.num_blocks = num_blocks;
  dl.post_norm = d.post_norm;
  dl.num_sms = h->num_sms;
  dl.eps = d.eps;
  std::memcpy(dl.rope_turn, h->rope_turn, sizeof(dl.rope_turn));
  dl.m_fc = &h->m_fc;
  dl.m_qkv = &h->m_qkv;
  dl.m_o = &h->m_o;
  dl.m_gate = &h->m_gate;
  dl.m_up = &h->m_up;
  dl.m_down = &h->m_down;
  dl.A = A;
  dl.n_valid = meta->n_valid;
  dl.valid_rows = meta->valid_rows;
  dl.valid_qsl = meta->valid_qsl;
  dl.pos = meta->pos;
  dl.slot = meta->slot;
  dl.gamma_in = h->w.gamma_in;
  dl.gamma_post = h->w.gamma_post;
  dl.gamma_final = h->w.gamma_final;
  dl.q_s = c.q_s;
  dl.k_cache = k_cache;
  dl.v_cache = v_cache;
  dl.x_s = c.x_s;
  dl.attn = c.attn;
  dl.z = z_out;
  dl.hidden_out = hidden_out;
  dl.scratch = at<void>(c.ws, c.L->dec);
  dl.bar = at<uint32_t>(c.ws, c.L->status + kBarrierWordsOffset);
  dl.status = c.status;
  int rc;
  if ((rc = launch_decode_layer(dl, 1, c.st)) != PE_OK) return rc;
  if ((rc = attention_step(c, Kd, B, meta, block_table, max_blocks, num_blocks, k_cache,
                           v_cache)) != PE_OK)
    return rc;
  return launch_decode_layer(dl, 2, c.st);
}

// The one-layer drafter over a batch of Kd draft rows per request (the handle's
// K for the parallel step, 1 for a pass of the autoregressive drafting): fc,
// QKV, RoPE + KV write, attention of the sample rows, O, MLP and the final norm
// into z_out [B*Kd][d].  hidden_out (nullable, fp32 [B*Kd][d]) receives the
// drafter's output hidden state of the sample rows: y (pre-norm) or the
// normalised output before rounding (post-norm).
int one_layer_step(const StepCtx& c, int Kd, int B, int T_in, const pe_meta* meta, const void* A,
                   const int32_t* block_table, int max_blocks, int num_blocks, void* k_cache,
                   void* v_cache, void* z_out, float* hidden_out) {
  pe_handle* h = c.h;
  const pe_dims& d = h->d;
  const int T_out = T_in + B * (Kd - 1);
  const int NS = B * Kd;
  const int QKV = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
  int rc, np = 1;
  if (c.bf && T_out <= kDecodeRows && NS <= kDecodeRows && c.L->dec)
    return decode_layer_step(c, Kd, B, T_in, meta, A, block_table, max_blocks, num_blocks,
                             k_cache, v_cache, z_out, hidden_out);
  if ((rc = fc_step(c, T_out, meta, A)) != PE_OK) return rc;
  // QKV (partial sums; RoPE adds them)
  Epilogue e = partial_epi(c, T_out, QKV);
  if ((rc = run_gemm(h, G_QKV, c.u, c.u_lo, T_out, meta->n_valid, e, c.ws, *c.L, c.st, true,
                     &np)) != PE_OK)
    return rc;
  // RoPE, KV write at the non-rejected slots, sample-row q and residual rows
  RopeArgs ra{};
  ra.T_out = T_out;
  ra.B = B;
  ra.K = Kd;
  ra.H = d.n_heads;
  ra.G = d.n_kv_heads;
  ra.hd = d.head_dim;
  ra.d = d.d;
  ra.bs = d.block_size;
  ra.num_blocks = num_blocks;
  ra.qkv = c.part;
  ra.n_parts = np;
  ra.part_stride = e.part_stride;
  ra.x = c.x;
  ra.n_valid = meta->n_valid;
  ra.valid_rows = meta->valid_rows;
  ra.valid_qsl = meta->valid_qsl;
  ra.pos = meta->pos;
  ra.slot = meta->slot;
  ra.k_cache = k_cache;
  ra.v_cache = v_cache;
  ra.q_s = c.q_s;
  ra.x_s = c.x_s;
  std::memcpy(ra.rope_turn, h->rope_turn, sizeof(ra.rope_turn));
  ra.status = c.status;
  if ((rc = launch_rope_kv(ra, c.dt, c.st)) != PE_OK) return rc;
  // paged attention of the sample rows
  AttnArgs aa{};
  aa.B = B;
  aa.K = Kd;
  aa.H = d.n_heads;
  aa.G = d.n_kv_heads;
  aa.hd = d.head_dim;
  aa.bs = d.block_size;
  aa.max_blocks = max_blocks;
  aa.num_blocks = num_blocks;
  plan_attention(B, d.n_kv_heads, Kd, d.n_heads, d.head_dim, max_blocks, d.block_size, h->num_sms,
                 aa.n_splits, aa.split_len, aa.cluster);
  aa.q = c.q_s;
  aa.k_cache = k_cache;
  aa.v_cache = v_cache;
  aa.block_table = block_table;
  aa.seq_len = meta->seq_len;
  aa.part_o = at<float>(c.ws, c.L->attn_part);
  aa.part_ml = reinterpret_cast<float*>(static_cast<char*>(c.ws) + c.L->attn_part +
                                        al256(static_cast<size_t>(aa.n_splits) * NS * d.n_heads *
                                              d.head_dim * sizeof(float)));
  aa.out = c.attn;
  aa.sink = static_cast<const float*>(h->w.attn_sink);
  aa.k_min = Kd;
  aa.status = c.status;
  if ((rc = launch_attention(aa, c.dt, c.st)) != PE_OK) return rc;
  // O projection (partial sums)
  e = partial_epi(c, NS, d.d);
  if ((rc = run_gemm(h, G_O, c.attn, nullptr, NS, nullptr, e, c.ws, *c.L, c.st, true, &np)) !=
      PE_OK)
    return rc;
  // r = x_s + attn W_o^T, and the MLP operand: post-norm a = RMSNorm(r;
  // gamma_post), which is also the MLP residual (kept as the fp32 value of the
  // pair); pre-norm m = RMSNorm(r), the residual being r itself
  if ((rc = step_norm(c, c.part, np, e.part_stride, c.x_s, d.post_norm ? nullptr : c.r,
                      h->w.gamma_post, 1, c.a, c.a_lo, d.post_norm ? c.a_f : nullptr, NS,
                      nullptr)) != PE_OK)
    return rc;
  const float* mlp_resid = d.post_norm ? (c.bf ? c.a_f : static_cast<const float*>(c.a)) : c.r;
  // SwiGLU: h = silu(gate) * up (a bf16 pair in bf16 mode)
  e = Epilogue();
  e.mode = c.bf ? EPI_SWIGLU_PAIR : EPI_SWIGLU;
  e.out = c.hm;
  e.out2 = c.h_lo;
  e.ld_out = d.inter;
  if ((rc = run_gemm(h, G_GATEUP, c.a, c.a_lo, NS, nullptr, e, c.ws, *c.L, c.st)) != PE_OK)
    return rc;
  // down projection (partial sums)
  e = partial_epi(c, NS, d.d);
  if ((rc = run_gemm(h, G_DOWN, c.hm, c.h_lo, NS, nullptr, e, c.ws, *c.L, c.st, true, &np)) !=
      PE_OK)
    return rc;
  // z = RMSNorm(y; gamma_final) with y = residual + h W_down^T: the LM head operand
  return step_norm(c, c.part, np, e.part_stride, mlp_resid,
                   hidden_out && !d.post_norm ? hidden_out : nullptr, h->w.gamma_final, 1, z_out,
                   nullptr, nullptr, NS, nullptr, hidden_out && d.post_norm ? hidden_out : nullptr);
}

// The N-layer drafter (N > 1): every layer runs over all non-rejected rows of
// each request, right-aligned in R rows (padding rows above them).
int layers_step(const StepCtx& c, int B, int T_in, const pe_meta* meta, const void* A,
                const int32_t* block_table, int max_blocks, int num_blocks, void* k_cache,
                void* v_cache, void* z_out) {
  pe_handle* h = c.h;
  const pe_dims& d = h->d;
  const Layout& L = *c.L;
  const int T_out = T_in + B * (d.K - 1);
  const int NS = B * d.K;
  const int Hd = d.n_heads * d.head_dim;
  const int QKV = (d.n_heads + 2 * d.n_kv_heads) * d.head_dim;
  const bool bf = c.bf;
  int rc, np = 1;
  if ((rc = fc_step(c, T_out, meta, A)) != PE_OK) return rc;
  const int R = layer_rows(h);
  const int NR = B * R;
  float* xl = at<float>(c.ws, L.xl);
  void* ul = at<void>(c.ws, L.ul);
  bf16_t* ul_lo = bf ? at<bf16_t>(c.ws, L.ul_lo) : nullptr;
  const size_t layer_elems =
      static_cast<size_t>(num_blocks) * d.n_kv_heads * d.block_size * d.head_dim;
  // rows no non-rejected row maps to keep finite values in the first layer
  if (cudaMemsetAsync(c.q_s, 0, static_cast<size_t>(NR) * Hd * esize(h), c.st) != cudaSuccess ||
      cudaMemsetAsync(c.x_s, 0, static_cast<size_t>(NR) * d.d * sizeof(float), c.st) != cudaSuccess)
    return PE_ERR_CUDA;
  for (int l = 0; l < h->n_layers; ++l) {
    const bool first = l == 0, last = l == h->n_layers - 1;
    const pe_layer_weights* lw = first ? nullptr : &h->more[l - 1].w;
    const void* g_post = first ? h->w.gamma_post : lw->gamma_post;
    const void* g_final = first ? h->w.gamma_final : lw->gamma_final;
    const float* sink = static_cast<const float*>(first ? h->w.attn_sink : lw->attn_sink);
    void* kc = static_cast<char*>(k_cache) + l * layer_elems * esize(h);
    void* vc = static_cast<char*>(v_cache) + l * layer_elems * esize(h);
    // QKV: the first layer over the non-rejected rows in order, later layers
    // over the right-aligned rows (partial sums; RoPE adds them)
    Epilogue e = partial_epi(c, first ? T_out : NR, QKV);
    if ((rc = first ? run_gemm(h, G_QKV, c.u, c.u_lo, T_out, meta->n_valid, e, c.ws, L, c.st, true,
                               &np)
                    : run_gemm(h, G_QKV, ul, ul_lo, NR, nullptr, e, c.ws, L, c.st, true, &np,
                               l)) != PE_OK)
      return rc;
    RopeArgs ra{};
    ra.T_out = T_out;
    ra.B = B;
    ra.K = R;
    ra.H = d.n_heads;
    ra.G = d.n_kv_heads;
    ra.hd = d.head_dim;
    ra.d = d.d;
    ra.bs = d.block_size;
    ra.num_blocks = num_blocks;
    ra.qkv = c.part;
    ra.n_parts = np;
    ra.part_stride = e.part_stride;
    ra.x = c.x;
    ra.n_valid = meta->n_valid;
    ra.valid_rows = meta->valid_rows;
    ra.valid_qsl = meta->valid_qsl;
    ra.pos = meta->pos;
    ra.slot = meta->slot;
    ra.k_cache = kc;
    ra.v_cache = vc;
    ra.q_s = c.q_s;
    ra.x_s = first ? c.x_s : nullptr;  // later layers' residual is already xl
    ra.padded_in = first ? 0 : 1;
    ra.must_fit = 1;
    std::memcpy(ra.rope_turn, h->rope_turn, sizeof(ra.rope_turn));
    ra.status = c.status;
    if ((rc = launch_rope_kv(ra, c.dt, c.st)) != PE_OK) return rc;
    AttnArgs aa{};
    aa.B = B;
    aa.K = R;
    aa.H = d.n_heads;
    aa.G = d.n_kv_heads;
    aa.hd = d.head_dim;
    aa.bs = d.block_size;
    aa.max_blocks = max_blocks;
    aa.num_blocks = num_blocks;
    plan_attention(B, d.n_kv_heads, R, d.n_heads, d.head_dim, max_blocks, d.block_size, h->num_sms,
                   aa.n_splits, aa.split_len, aa.cluster);
    aa.q = c.q_s;
    aa.k_cache = kc;
    aa.v_cache = vc;
    aa.block_table = block_table;
    aa.seq_len = meta->seq_len;
    aa.part_o = at<float>(c.ws, L.attn_part);
    aa.part_ml = reinterpret_cast<float*>(static_cast<char*>(c.ws) + L.attn_part +
                                          al256(static_cast<size_t>(aa.n_splits) * NR *
                                                d.n_heads * d.head_dim * sizeof(float)));
    aa.out = c.attn;
    aa.sink = sink;
    aa.k_min = d.K;
    aa.status = c.status;
    if ((rc = launch_attention(aa, c.dt, c.st)) != PE_OK) return rc;
    e = partial_epi(c, NR, d.d);
    if ((rc = run_gemm(h, G_O, c.attn, nullptr, NR, nullptr, e, c.ws, L, c.st, true, &np, l)) !=
        PE_OK)
      return rc;
    const float* resid = first ? c.x_s : xl;
    if ((rc = step_norm(c, c.part, np, e.part_stride, resid, d.post_norm ? nullptr : c.r, g_post, 1,
                        c.a, c.a_lo, d.post_norm ? c.a_f : nullptr, NR, nullptr)) != PE_OK)
      return rc;
    const float* mlp_resid = d.post_norm ? (bf ? c.a_f : static_cast<const float*>(c.a)) : c.r;
    e = Epilogue();
    e.mode = bf ? EPI_SWIGLU_PAIR : EPI_SWIGLU;
    e.out = c.hm;
    e.out2 = c.h_lo;
    e.ld_out = d.inter;
    if ((rc = run_gemm(h, G_GATEUP, c.a, c.a_lo, NR, nullptr, e, c.ws, L, c.st, true, nullptr,
                       l)) != PE_OK)
      return rc;
    e = partial_epi(c, NR, d.d);
    if ((rc = run_gemm(h, G_DOWN, c.hm, c.h_lo, NR, nullptr, e, c.ws, L, c.st, true, &np, l)) !=
        PE_OK)
      return rc;
    if (last) {
      // z: the final norm (pre-norm: the last layer's gamma_final) of the
      // sample rows, the last K of each request's R rows
      RowNormArgs n{};
      n.x = c.part;
      n.ld_x = d.d;
      n.n_parts = np;
      n.part_stride = e.part_stride;
      n.resid = mlp_resid;
      n.ld_resid = d.d;
      n.gamma = g_final;
      n.apply_norm = 1;
      n.out = z_out;
      n.ld_out = d.d;
      n.d = d.d;
      n.eps = d.eps;
      n.rows_cap = NS;
      n.in_group = R;
      n.out_group = d.K;
      return launch_rownorm(n, c.dt, c.st);
    }
    // the next layer's input: pre-norm y = residual + MLP (fp32) and its
    // QKV operand RMSNorm(y; gamma_in of the next layer); post-norm
    // RMSNorm(a + MLP; gamma_final), a bf16 pair that is also the residual
    if (d.post_norm) {
      rc = step_norm(c, c.part, np, e.part_stride, mlp_resid, nullptr, g_final, 1, ul, ul_lo, xl, NR,
                     nullptr);
    } else {
      rc = step_norm(c, c.part, np, e.part_stride, mlp_resid, xl, h->more[l].w.gamma_in, 1, ul,
                     ul_lo, nullptr, NR, nullptr);
    }
    if (rc != PE_OK) return rc;
  }
  return PE_OK;
}

// Workspace of pe_draft_autoregressive: a one-draft-row step's layout first
// (its status word is the call's), then pass 1's metadata (T_in rows), the
// metadata of a later pass (B rows), the drafter input rows, the fed-back hidden
// states (fp32) and z.
struct ArLayout {
  Layout layer;
  size_t m1[12], m2[12];
  size_t A, hidden, z, total;
};

ArLayout ar_layout(const pe_handle* h, int B, int T_in, int max_blocks) {
  ArLayout a{};
  a.layer = layout_of(h, B, T_in, max_blocks, 1);
  size_t off = a.layer.total;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = al256(off + bytes);
    return o;
  };
  auto meta = [&](size_t* m, int rows) {
    m[0] = take((B + 1) * sizeof(int32_t));            // out_qsl
    m[1] = take(rows * sizeof(int32_t));               // tok
    m[2] = take(rows * sizeof(int64_t));               // pos
    m[3] = take(rows);                                 // is_rejected
    m[4] = take(rows);                                 // is_masked
    m[5] = take(rows * sizeof(int32_t));               // hidden_src
    m[6] = take(rows * sizeof(int64_t));               // slot
    m[7] = take((B + 1) * sizeof(int32_t));            // valid_qsl
    m[8] = take(rows * sizeof(int32_t));               // valid_rows
    m[9] = take(sizeof(int32_t));                      // n_valid
    m[10] = take(B * sizeof(int32_t));                 // sample_idx
    m[11] = take(B * sizeof(int32_t));                 // seq_len
  };
  meta(a.m1, T_in);
  meta(a.m2, B);
  a.A = take(static_cast<size_t>(T_in) * 4 * h->d.d * esize(h));
  a.hidden = take(static_cast<size_t>(B) * h->d.d * sizeof(float));
  a.z = take(static_cast<size_t>(B) * h->d.d * esize(h));
  a.total = off;
  return a;
}

pe_meta meta_at(void* ws, const size_t* m) {
  pe_meta r;
  r.out_qsl = at<int32_t>(ws, m[0]);
  r.tok = at<int32_t>(ws, m[1]);
  r.pos = at<int64_t>(ws, m[2]);
  r.is_rejected = at<uint8_t>(ws, m[3]);
  r.is_masked = at<uint8_t>(ws, m[4]);
  r.hidden_src = at<int32_t>(ws, m[5]);
  r.slot = at<int64_t>(ws, m[6]);
  r.valid_qsl = at<int32_t>(ws, m[7]);
  r.valid_rows = at<int32_t>(ws, m[8]);
  r.n_valid = at<int32_t>(ws, m[9]);
  r.sample_idx = at<int32_t>(ws, m[10]);
  r.seq_len = at<int32_t>(ws, m[11]);
  return r;
}

}  // namespace

extern "C" {

int pe_create(const pe_dims* dims, const pe_weights* w, pe_handle** out) {
  if (!out) return PE_ERR_ARG;
  *out = nullptr;
  if (!dims || !w) return PE_ERR_ARG;
  const pe_dims& d = *dims;
  const bool bf = d.dtype == PE_DTYPE_BF16;
  if (check_dims(d) != PE_OK) return PE_ERR_UNSUPPORTED;
  const void* req[] = {w->emb, w->emb_mask, w->h_shared, w->gamma_stream};
  for (const void* p : req)
    if (!p || !aligned16(p)) return PE_ERR_ARG;
  // the layer's parameters: all of them, or none (a preparation-only handle)
  const void* layer[] = {w->w_fc,   w->w_qkv, w->w_o,    w->gamma_post, w->w_gate,
                         w->w_up,   w->w_down, w->gamma_final, w->w_lm};
  int n_layer = 0;
  for (const void* p : layer) {
    if (p && !aligned16(p)) return PE_ERR_ARG;
    n_layer += p ? 1 : 0;
  }
  const int n_all = static_cast<int>(sizeof(layer) / sizeof(layer[0]));
  if (n_layer != 0 && n_layer != n_all) return PE_ERR_ARG;
  const bool has_layer = n_layer == n_all;
  if (has_layer && !d.post_norm && (!w->gamma_in || !aligned16(w->gamma_in))) return PE_ERR_ARG;
  if (w->attn_sink && !aligned16(w->attn_sink)) return PE_ERR_ARG;
  // layers 2..N: every projection and gain (gamma_in pre-norm only), sinks optional
  const int n_layers = d.n_layers <= 0 ? 1 : d.n_layers;
  if (n_layers > 1) {
    if (!has_layer || !w->more_layers) return PE_ERR_ARG;
    for (int l = 0; l < n_layers - 1; ++l) {
      const pe_layer_weights& m = w->more_layers[l];
      const void* need[] = {m.w_qkv, m.w_o, m.gamma_post, m.w_gate, m.w_up, m.w_down,
                            m.gamma_final, d.post_norm ? m.w_qkv : m.gamma_in};
      for (const void* p : need)
        if (!p || !aligned16(p)) return PE_ERR_ARG;
      if (m.attn_sink && !aligned16(m.attn_sink)) return PE_ERR_ARG;
    }
  }
  // bf16: the GEMMs read the caller's tile-packed copy (pe_pack_weights)
  size_t packed_total = 0;
  std::vector<PackedMat> mats;
  if (bf && has_layer) {
    mats = packed_mats(d, w, &packed_total);
    if (!w->packed || (reinterpret_cast<uintptr_t>(w->packed) & 255u) ||
        w->packed_bytes < packed_total)
      return PE_ERR_ARG;
  }
  pe_handle* h = new (std::nothrow) pe_handle;
  if (!h) return PE_ERR_ARG;
  std::memset(h, 0, sizeof(*h));
  h->d = d;
  h->d.n_layers = n_layers;
  h->w = *w;
  h->w.more_layers = nullptr;  // the host array is read here only
  h->has_layer = has_layer;
  h->n_layers = n_layers;
  for (int l = 0; l < n_layers - 1; ++l) h->more[l].w = w->more_layers[l];
  h->num_sms = num_sms_of_current_device();
  if (h->num_sms <= 0) {
    delete h;
    return PE_ERR_CUDA;
  }
  // RoPE frequency i, theta^(-2i/hd) radians per position, as the fraction of a
  // turn per position in 64-bit fixed point (below 1/(2 pi) of a turn: no whole turns)
  for (int i = 0; i < d.head_dim / 2; ++i) {
    const double inv_freq = std::pow(static_cast<double>(d.rope_theta),
                                     -2.0 * static_cast<double>(i) / static_cast<double>(d.head_dim));
    const double turn = inv_freq / 6.283185307179586476925286766559;
    h->rope_turn[i] = static_cast<uint64_t>(std::ldexp(turn - std::floor(turn), 64));
  }
  if (bf && has_layer) {
    std::vector<CUtensorMap*> maps = {&h->m_fc, &h->m_qkv, &h->m_o,   &h->m_gate,
                                      &h->m_up, &h->m_down, &h->m_lm};
    for (int l = 0; l < n_layers - 1; ++l) {
      LayerSlot& ls = h->more[l];
      for (CUtensorMap* m : {&ls.m_qkv, &ls.m_o, &ls.m_gate, &ls.m_up, &ls.m_down}) maps.push_back(m);
    }
    for (size_t i = 0; i < mats.size(); ++i) {
      const void* P = static_cast<const char*>(w->packed) + mats[i].off;
      if (!encode_packed_weight_map(maps[i], P, mats[i].M, mats[i].K)) {
        delete h;
        return PE_ERR_CUDA;
      }
    }
  }
  *out = h;
  return PE_OK;
}

size_t pe_packed_weights_bytes(const pe_dims* dims) {
  if (!dims || check_dims(*dims) != PE_OK || dims->dtype != PE_DTYPE_BF16) return 0;
  size_t total = 0;
  packed_mats(*dims, nullptr, &total);
  return total;
}

int pe_pack_weights(const pe_dims* dims, const pe_weights* w, void* packed, size_t packed_bytes,
                    void* stream) {
  NvtxRange nvtx("pe_pack_weights");
  if (!dims || !w || !packed) return PE_ERR_ARG;
  if (check_dims(*dims) != PE_OK || dims->dtype != PE_DTYPE_BF16) return PE_ERR_UNSUPPORTED;
  if (dims->n_layers > 1 && !w->more_layers) return PE_ERR_ARG;
  size_t total = 0;
  const std::vector<PackedMat> mats = packed_mats(*dims, w, &total);
  if ((reinterpret_cast<uintptr_t>(packed) & 255u) || packed_bytes < total) return PE_ERR_ARG;
  for (const PackedMat& m : mats)
    if (!m.W || !aligned16(m.W)) return PE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (const PackedMat& m : mats) {
    const int rc = pack_weight(m.W, m.M, m.K, static_cast<char*>(packed) + m.off, st);
    if (rc != PE_OK) return rc;
  }
  return PE_OK;
}

void pe_destroy(pe_handle* h) { delete h; }

size_t pe_workspace_bytes(const pe_handle* h, int max_batch, int max_rows_in,
                          int max_blocks_per_seq) {
  if (!h || max_batch < 1 || max_rows_in < 1 || max_blocks_per_seq < 1) return 0;
  const Layout a = layout_of(h, max_batch, max_rows_in, max_blocks_per_seq);
  const Layout b = layout_argmax(h, max_batch * h->d.K);
  return std::max(a.total, b.total);
}

int pe_prepare_inputs(pe_handle* h, int B, int T_in, const int32_t* qsl, const int32_t* prev_tok,
                      const int64_t* prev_pos, const int32_t* accepted, const int32_t* bonus,
                      const int32_t* block_table, int max_blocks, int num_blocks,
                      const void* H_tgt, const pe_meta* meta, void* G_out, void* E_out,
                      void* A_out, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("pe_prepare_inputs");
  if (!h || B < 1 || T_in < B || max_blocks < 1 || num_blocks < 1 || !qsl || !prev_tok ||
      !prev_pos || !accepted || !bonus || !block_table || !H_tgt || !ws)
    return PE_ERR_ARG;
  if (check_meta(meta) != PE_OK) return PE_ERR_ARG;
  if (ws_bytes < 256 || !aligned16(ws) || !aligned16(H_tgt)) return PE_ERR_ARG;
  if ((G_out && !aligned16(G_out)) || (E_out && !aligned16(E_out)) || (A_out && !aligned16(A_out)))
    return PE_ERR_ARG;
  const pe_dims& d = h->d;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = at<uint32_t>(ws, 0);
  // the status word and the decode layer's barrier words
  if (cudaMemsetAsync(status, 0, 256, st) != cudaSuccess) return PE_ERR_CUDA;
  MetaLaunch ml;
  ml.B = B;
  ml.T_in = T_in;
  ml.K = d.K;
  ml.mask_id = d.mask_id;
  ml.bs = d.block_size;
  ml.max_blocks = max_blocks;
  ml.num_blocks = num_blocks;
  ml.vocab = d.vocab;
  ml.qsl = qsl;
  ml.prev_tok = prev_tok;
  ml.prev_pos = prev_pos;
  ml.accepted = accepted;
  ml.bonus = bonus;
  ml.block_table = block_table;
  ml.meta = *meta;
  ml.status = status;
  int rc = launch_meta(ml, st);
  if (rc != PE_OK) return rc;
  const int T_out = T_in + B * (d.K - 1);
  if (G_out || E_out) {
    GatherArgs g{};
    g.T_out = T_out;
    g.T_in = T_in;
    g.d = d.d;
    g.vocab = d.vocab;
    g.hidden_src = meta->hidden_src;
    g.tok = meta->tok;
    g.is_masked = meta->is_masked;
    g.H_tgt = H_tgt;
    g.h_shared = h->w.h_shared;
    g.emb = h->w.emb;
    g.emb_mask = h->w.emb_mask;
    g.G = G_out;
    g.E = E_out;
    g.status = status;
    rc = launch_gather(g, d.dtype, h->num_sms, st);
    if (rc != PE_OK) return rc;
  }
  if (A_out) {
    InputArgs ia{};
    ia.T_out = T_out;
    ia.T_in = T_in;
    ia.d = d.d;
    ia.vocab = d.vocab;
    ia.eps = d.eps;
    ia.n_valid = meta->n_valid;
    ia.valid_rows = meta->valid_rows;
    ia.hidden_src = meta->hidden_src;
    ia.tok = meta->tok;
    ia.is_masked = meta->is_masked;
    ia.H_tgt = H_tgt;
    ia.h_shared = h->w.h_shared;
    ia.emb = h->w.emb;
    ia.emb_mask = h->w.emb_mask;
    ia.gamma_stream = h->w.gamma_stream;
    ia.A = A_out;
    ia.status = status;
    // small batches: the input kernel indexes its rows itself and runs beside
    // the metadata kernel (no gather kernel between them)
    ia.self_index = (B <= kSelfIndexMaxBatch && !(G_out || E_out)) ? 1 : 0;
    ia.B = B;
    ia.K = d.K;
    ia.qsl = qsl;
    ia.prev_tok = prev_tok;
    ia.accepted = accepted;
    ia.bonus = bonus;
    rc = launch_input(ia, d.dtype, st);
    if (rc != PE_OK) return rc;
  }
  return PE_OK;
}

int pe_draft_step(pe_handle* h, int B, int T_in, const pe_meta* meta, const void* A,
                  const int32_t* block_table, int max_blocks, int num_blocks, void* k_cache,
                  void* v_cache, void* z_out, void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("pe_draft_step");
  if (!h || !h->has_layer || B < 1 || T_in < B || max_blocks < 1 || num_blocks < 1 || !A ||
      !block_table || !k_cache || !v_cache || !z_out || !ws)
    return PE_ERR_ARG;
  if (check_meta(meta) != PE_OK) return PE_ERR_ARG;
  if (!aligned16(A) || !aligned16(z_out) || !aligned16(ws)) return PE_ERR_ARG;
  const pe_dims& d = h->d;
  const Layout L = layout_of(h, B, T_in, max_blocks);
  if (ws_bytes < L.total) return PE_ERR_ARG;
  const StepCtx c = make_ctx(h, L, ws, static_cast<cudaStream_t>(stream));
  if (h->n_layers <= 1)
    return one_layer_step(c, d.K, B, T_in, meta, A, block_table, max_blocks, num_blocks, k_cache,
                          v_cache, z_out, nullptr);
  return layers_step(c, B, T_in, meta, A, block_table, max_blocks, num_blocks, k_cache, v_cache,
                     z_out);
}

size_t pe_autoregressive_workspace_bytes(const pe_handle* h, int max_batch, int max_rows_in,
                                         int max_blocks_per_seq) {
  if (!h || max_batch < 1 || max_rows_in < max_batch || max_blocks_per_seq < 1) return 0;
  return ar_layout(h, max_batch, max_rows_in, max_blocks_per_seq).total;
}

int pe_draft_autoregressive(pe_handle* h, int B, int T_in, const int32_t* qsl,
                            const int32_t* prev_tok, const int64_t* prev_pos,
                            const int32_t* accepted, const int32_t* bonus,
                            const int32_t* block_table, int max_blocks, int num_blocks,
                            const void* H_tgt, void* k_cache, void* v_cache, int32_t* draft_tokens,
                            float* logits, float* hidden_out, void* ws, size_t ws_bytes,
                            void* stream) {
  NvtxRange nvtx("pe_draft_autoregressive");
  if (!h || !h->has_layer || B < 1 || T_in < B || max_blocks < 1 || num_blocks < 1 || !qsl ||
      !prev_tok || !prev_pos || !accepted || !bonus || !block_table || !H_tgt || !k_cache ||
      !v_cache || !draft_tokens || !ws)
    return PE_ERR_ARG;
  if (h->n_layers > 1) return PE_ERR_UNSUPPORTED;
  if (!aligned16(ws) || !aligned16(H_tgt)) return PE_ERR_ARG;
  const pe_dims& d = h->d;
  const ArLayout AL = ar_layout(h, B, T_in, max_blocks);
  if (ws_bytes < AL.total) return PE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const StepCtx c = make_ctx(h, AL.layer, ws, st);
  if (cudaMemsetAsync(c.status, 0, 256, st) != cudaSuccess) return PE_ERR_CUDA;
  const pe_meta m1 = meta_at(ws, AL.m1);
  const pe_meta m2 = meta_at(ws, AL.m2);
  void* A = at<void>(ws, AL.A);
  float* hidden = at<float>(ws, AL.hidden);
  void* z = at<void>(ws, AL.z);
  unsigned long long* keys = at<unsigned long long>(ws, AL.layer.amax);
  // the LM head of pass k: draft k of every request (and its logits, if asked)
  auto lm_pass = [&](int k) {
    if (launch_zero_keys(keys, B, st) != PE_OK) return PE_ERR_CUDA;
    Epilogue e;
    e.mode = EPI_ARGMAX;
    e.amax = keys;
    e.logits = logits ? logits + static_cast<size_t>(k - 1) * d.vocab : nullptr;
    e.ld_logits = d.K * d.vocab;
    int rc = run_gemm(h, G_LM, z, nullptr, B, nullptr, e, ws, AL.layer, st);
    if (rc != PE_OK) return rc;
    rc = launch_argmax_finalize(keys, B, draft_tokens + (k - 1), st, d.K);
    if (rc != PE_OK || !hidden_out) return rc;
    // this pass's hidden states into column k - 1 of hidden_out [B][K][d]
    const size_t row = static_cast<size_t>(d.d) * sizeof(float);
    return cudaMemcpy2DAsync(hidden_out + static_cast<size_t>(k - 1) * d.d, d.K * row, hidden, row,
                             row, B, cudaMemcpyDeviceToDevice, st) == cudaSuccess
               ? PE_OK
               : PE_ERR_CUDA;
  };
  // pass 1: the parallel step with one draft row per request (its NTP row)
  MetaLaunch ml;
  ml.B = B;
  ml.T_in = T_in;
  ml.K = 1;
  ml.mask_id = d.mask_id;
  ml.bs = d.block_size;
  ml.max_blocks = max_blocks;
  ml.num_blocks = num_blocks;
  ml.vocab = d.vocab;
  ml.qsl = qsl;
  ml.prev_tok = prev_tok;
  ml.prev_pos = prev_pos;
  ml.accepted = accepted;
  ml.bonus = bonus;
  ml.block_table = block_table;
  ml.meta = m1;
  ml.status = c.status;
  int rc = launch_meta(ml, st);
  if (rc != PE_OK) return rc;
  InputArgs ia{};
  ia.T_out = T_in;
  ia.T_in = T_in;
  ia.d = d.d;
  ia.vocab = d.vocab;
  ia.eps = d.eps;
  ia.n_valid = m1.n_valid;
  ia.valid_rows = m1.valid_rows;
  ia.hidden_src = m1.hidden_src;
  ia.tok = m1.tok;
  ia.is_masked = m1.is_masked;
  ia.H_tgt = H_tgt;
  ia.h_shared = h->w.h_shared;
  ia.emb = h->w.emb;
  ia.emb_mask = h->w.emb_mask;
  ia.gamma_stream = h->w.gamma_stream;
  ia.A = A;
  ia.status = c.status;
  if ((rc = launch_input(ia, d.dtype, st)) != PE_OK) return rc;
  if ((rc = one_layer_step(c, 1, B, T_in, &m1, A, block_table, max_blocks, num_blocks, k_cache,
                           v_cache, z, hidden)) != PE_OK)
    return rc;
  if ((rc = lm_pass(1)) != PE_OK) return rc;
  // passes 2..K: one row per request, fed its own hidden state and last draft
  for (int k = 2; k <= d.K; ++k) {
    ArInputArgs ai{};
    ai.B = B;
    ai.K = d.K;
    ai.k = k;
    ai.d = d.d;
    ai.vocab = d.vocab;
    ai.bs = d.block_size;
    ai.max_blocks = max_blocks;
    ai.num_blocks = num_blocks;
    ai.eps = d.eps;
    ai.pos1 = m1.pos;
    ai.sample1 = m1.sample_idx;
    ai.drafts = draft_tokens;
    ai.hidden = hidden;
    ai.block_table = block_table;
    ai.emb = h->w.emb;
    ai.gamma_stream = h->w.gamma_stream;
    ai.meta = m2;
    ai.A = A;
    ai.status = c.status;
    if ((rc = launch_ar_input(ai, d.dtype, st)) != PE_OK) return rc;
    if ((rc = one_layer_step(c, 1, B, B, &m2, A, block_table, max_blocks, num_blocks, k_cache,
                             v_cache, z, hidden)) != PE_OK)
      return rc;
    if ((rc = lm_pass(k)) != PE_OK) return rc;
  }
  return PE_OK;
}

int pe_argmax(pe_handle* h, const void* z, int n_rows, int32_t* draft_tokens, float* logits,
              void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("pe_argmax");
  if (!h || !h->has_layer || !z || n_rows < 1 || !draft_tokens || !ws) return PE_ERR_ARG;
  if (!aligned16(z) || !aligned16(ws)) return PE_ERR_ARG;
  const Layout L = layout_argmax(h, n_rows);
  if (ws_bytes < L.total) return PE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned long long* keys = at<unsigned long long>(ws, L.amax);
  if (launch_zero_keys(keys, n_rows, st) != PE_OK) return PE_ERR_CUDA;
  Epilogue e;
  e.mode = EPI_ARGMAX;
  e.amax = keys;
  e.logits = logits;
  e.ld_logits = h->d.vocab;
  int rc = run_gemm(h, G_LM, z, nullptr, n_rows, nullptr, e, ws, L, st);
  if (rc != PE_OK) return rc;
  return launch_argmax_finalize(keys, n_rows, draft_tokens, st);
}

int pe_test_bounded_wait(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < 256 || !aligned16(ws)) return PE_ERR_ARG;
  return launch_bounded_wait(static_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream));
}

size_t pe_test_projection_workspace(const pe_handle* h, int which, int n_rows) {
  const bool argmax = (which & PE_PROJ_ARGMAX) != 0;
  which &= ~(PE_PROJ_PERSISTENT | PE_PROJ_PAIR | PE_PROJ_PARTIAL | PE_PROJ_ARGMAX);
  if (!h || which < 0 || which >= G_COUNT || n_rows < 1) return 0;
  return layout_projection(h, which, n_rows, argmax).total;
}

int pe_test_projection(pe_handle* h, int which, const void* X, int n_rows, void* out, void* ws,
                       size_t ws_bytes, void* stream) {
  const bool persistent = (which & PE_PROJ_PERSISTENT) != 0;
  const bool pair = (which & PE_PROJ_PAIR) != 0;
  const bool partial = (which & PE_PROJ_PARTIAL) != 0;
  const bool argmax = (which & PE_PROJ_ARGMAX) != 0;
  which &= ~(PE_PROJ_PERSISTENT | PE_PROJ_PAIR | PE_PROJ_PARTIAL | PE_PROJ_ARGMAX);
  if (partial && which == G_GATEUP) return PE_ERR_ARG;
  if (argmax && (which != G_LM || partial || pair)) return PE_ERR_ARG;
  if (!h || !h->has_layer || which < 0 || which >= G_COUNT || n_rows < 1 || !X || !out || !ws)
    return PE_ERR_ARG;
  if (!aligned16(X) || !aligned16(ws)) return PE_ERR_ARG;
  if (pair && !is_bf16(h)) return PE_ERR_UNSUPPORTED;
  const Layout L = layout_projection(h, which, n_rows, argmax);
  if (ws_bytes < L.total) return PE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const GemmShape s = gemm_shape(h, which);
  if (argmax) {
    unsigned long long* keys = at<unsigned long long>(ws, L.amax);
    if (launch_zero_keys(keys, n_rows, st) != PE_OK) return PE_ERR_CUDA;
    Epilogue e;
    e.mode = EPI_ARGMAX;
    e.amax = keys;
    e.logits = static_cast<float*>(out);
    e.ld_logits = s.M;
    const int rc = run_gemm(h, which, X, nullptr, n_rows, nullptr, e, ws, L, st, !persistent);
    if (rc != PE_OK) return rc;
    return launch_argmax_finalize(keys, n_rows, at<int32_t>(ws, L.tok), st);
  }
  Epilogue e;
  e.mode = which == G_GATEUP ? EPI_SWIGLU : partial ? EPI_PARTIAL_F32 : EPI_STORE_F32;
  e.out = out;
  e.ld_out = s.M;
  e.part_stride = static_cast<size_t>(n_rows) * s.M;
  const void* X_lo =
      pair ? static_cast<const void*>(static_cast<const bf16_t*>(X) +
                                      static_cast<size_t>(n_rows) * s.K)
           : nullptr;
  return run_gemm(h, which, X, X_lo, n_rows, nullptr, e, ws, L, st, !persistent);
}

int pe_read_status(const pe_handle* h, void* ws, uint32_t* status, int clear, void* stream) {
  (void)h;  // the word lives in ws; handle-free calls pass NULL
  if (!ws || !status) return PE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return PE_ERR_CUDA;
  if (clear && cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return PE_ERR_CUDA;
  *status = v;
  if (v & PE_ST_TIMEOUT) return PE_ERR_TIMEOUT;
  return v ? PE_ERR_DEVICE_INPUT : PE_OK;
}

const char* pe_status_string(int code) {
  switch (code) {
    case PE_OK: return "ok";
    case PE_ERR_ARG: return "invalid argument (null pointer, size, alignment or workspace too small)";
    case PE_ERR_UNSUPPORTED: return "unsupported dimensions";
    case PE_ERR_CUDA: return "CUDA runtime or launch error";
    case PE_ERR_DEVICE_INPUT: return "the device found out-of-range inputs (see the status bits)";
    case PE_ERR_TIMEOUT: return "a bounded device wait expired";
    default: return "unknown status code";
  }
}

}  // extern "C"

// Read-only views of a handle for other translation units of the library.
namespace pe {
const pe_dims* handle_dims(const pe_handle* h) { return &h->d; }
const CUtensorMap* handle_lm_map(const pe_handle* h) { return &h->m_lm; }
int handle_num_sms(const pe_handle* h) { return h->num_sms; }
const void* handle_w_lm(const pe_handle* h) { return h->w.w_lm; }
bool handle_has_layer(const pe_handle* h) { return h->has_layer; }
}  // namespace pe
