// The decoder layer of a decode-sized step as two persistent kernels.
//
// With at most 16 token rows every projection of the layer streams its weight
// matrix from DRAM.  Run as separate kernels (fc, row norm, QKV, RoPE, O, row
// norm, gate/up, down, final norm) each boundary costs a launch, a pipeline
// fill and a drain, and the DRAM stream stops in between.  Here one launch
// covers fc -> QKV -> RoPE/KV write and a second covers O -> gate/up -> down
// -> final norm (attention runs between them as its own kernel):
//
//   * Every CTA (2 per SM, all resident) owns at most one work item of each
//     projection: one 128-row weight tile and one share of its reduction
//     dimension.  It stores the partial product of its share (fp32); the
//     elementwise stage after the projection adds the shares in order.
//   * Stages hand off through grid barriers in global memory (arrival counts,
//     bounded waits).  A projection's weight boxes depend on nothing, so the
//     TMA warp issues its first ring stages before it waits for the barrier that
//     releases the token operand: the next projection's weights stream while the
//     stage before it finishes.
//   * A row norm before a projection needs the whole row's sum of squares.  The
//     elementwise stage writes the un-normalised operand (x * gamma, as a bf16
//     pair) and per-chunk sums of squares; the stage after the projection scales
//     each row by 1/rms (the projection is linear in its operand).
//
// Warp roles: warp 0 issues TMA, one thread of warp 1 issues tcgen05.mma into
// TMEM (128 x 16 fp32 accumulator), warps 2-5 read the accumulator, store the
// partial tile, and run the elementwise stages.  Every wait is bounded: a wait
// that runs out sets PE_ST_TIMEOUT and a global abort word, and every CTA
// leaves.
#include <algorithm>
#include <cstring>

#include "pe_common.cuh"
#include "pe_internal.h"
#include "pe_prep.h"

namespace pe {

namespace {

constexpr int kThreads = 192;
// The grid barriers need every CTA of the grid resident at once.  Three CTAs
// fit an SM, but the grid takes two per SM: with every slot needed, a single
// SM slot held up elsewhere once in a while left the last CTA unscheduled and
// the others waiting at the first barrier until the bounded wait ran out
// (measured: a few of 60 replays of a 7-pass autoregressive graph).
constexpr int kCtasPerSm = 2;
constexpr int kBM = 128;                          // weight rows per tile (MMA M)
constexpr int kBK = 64;                           // reduction elements per k-block
// Ring stages: the first ones of each projection are issued before the wait for
// its token operand, so a deeper ring keeps more of the next weights in flight
// across a stage boundary (two CTAs of five 20 KB stages fit an SM).
constexpr int kSlots = 5;
constexpr uint32_t kABytes = kBM * kBK * 2;       // 16 KB weight box
constexpr uint32_t kBBytes = kDecodeRows * 128;   // 2 KB token box (16 rows)
constexpr uint32_t kSlotBytes = kABytes + 2 * kBBytes;
constexpr size_t kSmemBytes = kSlots * kSlotBytes + 1024;
// kCtasPerSm CTAs fit an SM's 228 KB of shared memory: the ring, under 1 KB of
// static shared memory and the 1 KB the system reserves per CTA.  (The
// occupancy query answers 1 for tcgen05 kernels like this one whatever their
// size, so the fit is this arithmetic.)
static_assert(kCtasPerSm * (kSmemBytes + 2048) <= 228 * 1024, "decode CTAs must fit an SM");
constexpr int kChunk = 128;                       // features per elementwise unit
constexpr int kMaxGemm = 3;
constexpr uint32_t kTmemCols = 32;

// Barrier words (uint32) in the workspace header, after the status word.
enum : int {
  BW_PART1 = 0,     // part 1: 0 fc done, 1 operand written, 2 QKV done, 3 CTAs done
  BW_PART2 = 4,     // part 2: 4 O done, 5 operand, 6 gate/up, 7 SwiGLU, 8 down, 9 y, 10 done
  BW_EPOCH1 = 12,   // completed launches of part 1 / part 2
  BW_EPOCH2 = 13,
  BW_ABORT = 14,    // set by a CTA whose wait ran out: every other CTA leaves
  BW_COUNT = 16,
};
static_assert(BW_EPOCH1 == 12, "PE_TEST_DECODE_EPOCH_BYTE names word 12 of the header");

struct DecGemm {
  int M, K, num_kb, kbps, splits, m_tiles, n_mats, bpair, items;
  float* out;       // partial tiles: out[((mat * splits + ks) * 16 + t) * M + f]
};

struct DecParams {
  CUtensorMap mapA[kMaxGemm][2];  // packed weights of each projection (two for gate/up)
  CUtensorMap mapB[kMaxGemm][2];  // token operand (hi, lo; lo = hi when not a pair)
  DecGemm g[kMaxGemm];
  int n_gemm;
  int d, H, G, hd, inter, K, B, bs, num_blocks, post_norm;
  float eps;
  int rows_cap;            // token rows: T_out (part 1) or B*K (part 2)
  const int* n_rows_dev;   // part 1: live rows (n_valid); part 2: NULL
  const int32_t* valid_rows;
  const int32_t* valid_qsl;
  const int64_t* pos;
  const int64_t* slot;
  float* x_s;              // [B*K][d] residual rows of the sample rows
  bf16* op_hi;             // projection operand pair [16][d]
  bf16* op_lo;
  bf16* h_hi;              // SwiGLU product pair [16][I]
  bf16* h_lo;
  float* r;                // [16][d] attention residual sum
  float* y;                // [16][d] MLP residual sum
  float* ss;               // [16][64] sums of squares per (row, 128-feature chunk)
  float* ss2;              // [16][64] (final norm)
  const bf16* gamma_a;     // part 1: gamma_in; part 2: gamma_post
  const bf16* gamma_b;     // part 2: gamma_final
  bf16* q_s;
  bf16* k_cache;
  bf16* v_cache;
  bf16* z;                 // [B*K][d]
  float* hidden_out;       // [B*K][d], nullable: the state handed to the next pass
  uint32_t* bar;           // BW_COUNT barrier words
  uint32_t* status;
  uint64_t rope_turn[64];
};

PE_DEV uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait until barrier word w has reached `target` arrivals (wrap-safe compare).
// Bounded; gives up early when another CTA has aborted.
PE_DEV bool grid_wait(const DecParams& p, int w, uint32_t target) {
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 0;; ++i) {
    if (static_cast<int32_t>(ld_acquire(p.bar + w) - target) >= 0) return true;
    if ((i & 63u) == 63u) {
      if (ld_acquire(p.bar + BW_ABORT)) return false;
      if (globaltimer() - t0 > kWaitNs) return false;
    }
  }
}

PE_DEV void grid_arrive(const DecParams& p, int w) {
  __threadfence();
  atomicAdd(p.bar + w, 1u);
}

// A wait that ran out: the status bit, the abort word every CTA polls, and the
// first place that gave up (header word 15: part << 16 | where << 8 | block, in
// words 32.. the block, the barrier word, its count and the target).
PE_DEV void abort_all(const DecParams& p, int part, int where, uint32_t word = 0,
                      uint32_t target = 0) {
  set_status(p.status, PE_ST_TIMEOUT);
  if (atomicCAS(p.bar + 15, 0u, 1u + ((part << 16) | (where << 8))) == 0u) {
    p.bar[16] = blockIdx.x;
    p.bar[17] = word;
    p.bar[18] = word < 16 ? p.bar[word] : 0u;
    p.bar[19] = target;
  }
  atomicExch(p.bar + BW_ABORT, 1u);
}

// Generic-proxy writes of other CTAs (seen through an acquire) before this
// thread's TMA (async-proxy) reads of the same global memory.
PE_DEV void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The packed weight box of tile row m at k-block kb (beyond K: past the last
// block, which TMA fills with zeros).
PE_DEV void weight_box(const DecGemm& g, int m, int kb, int& cx, int& cy) {
  const int k_atoms = (g.K + kBK - 1) / kBK;
  cx = 0;
  cy = (kb < k_atoms ? m * k_atoms + kb : g.m_tiles * k_atoms) * kBM;
}

struct Item {
  int mat, m, ks, kb0, kb1;
};

PE_DEV bool item_of(const DecGemm& g, int it, Item& out) {
  if (it >= g.items) return false;
  const int per_mat = g.m_tiles * g.splits;
  out.mat = it / per_mat;
  const int rem = it - out.mat * per_mat;
  out.m = rem / g.splits;
  out.ks = rem - out.m * g.splits;
  out.kb0 = out.ks * g.kbps;
  out.kb1 = min(g.num_kb, out.kb0 + g.kbps);
  return out.kb0 < out.kb1;
}

// Sums of the partial tiles of projection g (matrix `mat`) at row t for N
// features f[i] (f[i] < 0: none, 0 returned; a feature of matrix 1 may also be
// given as f + splits * 16 * M with mat = 0).  The shares are added in split
// order; the loads of W shares of every feature are issued together.
template <int N, int W>
PE_DEV void sum_parts(const DecGemm& g, int mat, int t, const int (&f)[N], float (&out)[N]) {
  const float* p = g.out + (static_cast<size_t>(mat) * g.splits * kDecodeRows + t) * g.M;
  const size_t stride = static_cast<size_t>(kDecodeRows) * g.M;
#pragma unroll
  for (int i = 0; i < N; ++i) out[i] = 0.f;
  for (int k0 = 0; k0 < g.splits; k0 += W) {
    float v[N][W];
#pragma unroll
    for (int i = 0; i < N; ++i)
#pragma unroll
      for (int k = 0; k < W; ++k)
        v[i][k] = (f[i] >= 0 && k0 + k < g.splits) ? p[(k0 + k) * stride + f[i]] : 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i)
#pragma unroll
      for (int k = 0; k < W; ++k)
        if (k0 + k < g.splits) out[i] += v[i][k];
  }
}

// Row norms in two steps, so that the loads go out beside the others: this
// lane's share of row t's per-chunk sums of squares (chunks lane and lane + 32),
// then 1 / rms from the warp's shares.
PE_DEV float ss_share(const float* ss, int t, int nc) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  if (lane < nc) s += ss[t * 64 + lane];
  if (lane + 32 < nc) s += ss[t * 64 + lane + 32];
  return s;
}

PE_DEV float inv_rms(float share, int d, float eps) {
  const float s = warp_sum(share);
  return 1.0f / sqrtf(s / static_cast<float>(d) + eps);
}

// The sample row (r * K + k) non-rejected row v is, or -1: one of the last K
// non-rejected rows of its request.  One warp-wide lookup (B <= 32); every lane
// of the warp calls it with the same v.
PE_DEV int sample_of(const DecParams& p, int v) {
  const int lane = threadIdx.x & 31;
  int v0 = 0, v1 = 0;
  if (lane < p.B) {
    v0 = p.valid_qsl[lane];
    v1 = p.valid_qsl[lane + 1];
  }
  const uint32_t hit = __ballot_sync(0xffffffffu, lane < p.B && v >= v0 && v < v1);
  if (!hit) return -1;
  const int r = __ffs(static_cast<int>(hit)) - 1;
  const int k = v - (__shfl_sync(0xffffffffu, v1, r) - p.K);
  return k >= 0 && k < p.K ? r * p.K + k : -1;
}

PE_DEV void store_pair(bf16* hi, bf16* lo, size_t i, float v) {
  const bf16 h = __float2bfloat16_rn(v);
  hi[i] = h;
  lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
}

// Sums of x[i] over the 128 elementwise threads (4 warps); `red` holds 4 * N floats.
template <int N>
PE_DEV void sum128(float (&x)[N], float* red) {
  const int ew = (threadIdx.x >> 5) - 2, lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < N; ++i) x[i] = warp_sum(x[i]);
  named_bar_sync(2, 128);
  if (lane == 0)
#pragma unroll
    for (int i = 0; i < N; ++i) red[i * 4 + ew] = x[i];
  named_bar_sync(2, 128);
#pragma unroll
  for (int i = 0; i < N; ++i) x[i] = red[i * 4] + red[i * 4 + 1] + red[i * 4 + 2] + red[i * 4 + 3];
}

// ---------------------------------------------------------------- elementwise stages
//
// The units of a stage are (row, group of up to kMaxCG consecutive 128-feature
// chunks): groups wide enough that the units fit one round of the grid, each
// thread one feature of every chunk of its unit, all loads issued together.
constexpr int kMaxCG = 2;

PE_DEV int chunks_per_unit(int rows, int nc) {
  const int cg = (rows * nc + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);
  return min(max(cg, 1), kMaxCG);
}

// Features of unit chunk group c0 .. c0 + cg - 1 for this thread (j), -1 past
// the group or past M.
PE_DEV void unit_features(int c0, int cg, int M, int (&f)[kMaxCG]) {
  const int j = threadIdx.x - 64;
#pragma unroll
  for (int i = 0; i < kMaxCG; ++i) {
    const int ff = (c0 + i) * kChunk + j;
    f[i] = (i < cg && ff < M) ? ff : -1;
  }
}

// Part 1, after fc: x = the fc shares' sum for non-rejected row v; the QKV
// operand (x * gamma_in pre-norm, x post-norm) as a bf16 pair; x of the sample
// rows (the attention residual); per-chunk sums of squares of x (pre-norm).
PE_DEV void stage_after_fc(const DecParams& p, int n_rows, float* red, int s_first) {
  const int nc = (p.d + kChunk - 1) / kChunk;
  const int cg = chunks_per_unit(n_rows, nc);
  const int ngr = (nc + cg - 1) / cg;
  for (int u = blockIdx.x; u < n_rows * ngr; u += gridDim.x) {
    const int v = u / ngr, c0 = (u - v * ngr) * cg;
    int f[kMaxCG];
    unit_features(c0, cg, p.d, f);
    float x[kMaxCG], sq[kMaxCG];
    sum_parts<kMaxCG, 16>(p.g[0], 0, v, f, x);
    const int s = u == static_cast<int>(blockIdx.x) ? s_first : sample_of(p, v);
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i) {
      sq[i] = 0.f;
      if (f[i] < 0) continue;
      const float opv = p.post_norm ? x[i] : x[i] * __bfloat162float(p.gamma_a[f[i]]);
      store_pair(p.op_hi, p.op_lo, static_cast<size_t>(v) * p.d + f[i], opv);
      if (s >= 0) p.x_s[static_cast<size_t>(s) * p.d + f[i]] = x[i];
      sq[i] = x[i] * x[i];
    }
    if (!p.post_norm) {
      sum128(sq, red);
      if (threadIdx.x == 64)
#pragma unroll
        for (int i = 0; i < kMaxCG; ++i)
          if (i < cg && c0 + i < nc) p.ss[v * 64 + c0 + i] = sq[i];
    }
  }
}

// The metadata of a warp's first RoPE unit (row v, head hh): the row's index in
// the step's row arrays, its position and cache slot, and its sample row (q
// heads); and this lane's two RoPE frequencies (a per-lane index into the
// kernel parameters reads the constant bank lane by lane).  Loaded while fc
// streams, so the RoPE stage waits only for its sums.
struct RopeMeta {
  int u, o, s;
  int64_t pos, slot;
  uint64_t turn[2];
};

PE_DEV RopeMeta rope_meta(const DecParams& p, int n_rows) {
  const int heads = p.H + 2 * p.G;
  RopeMeta m;
  m.u = blockIdx.x * 4 + ((threadIdx.x >> 5) - 2);
  m.o = 0;
  m.s = -1;
  m.pos = 0;
  m.slot = PE_PADDING_SLOT_ID;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 2; ++q) m.turn[q] = lane + 32 * q < p.hd / 2 ? p.rope_turn[lane + 32 * q] : 0ull;
  if (m.u < n_rows * heads) {
    const int v = m.u / heads, hh = m.u - (m.u / heads) * heads;
    m.o = p.valid_rows[v];
    m.s = hh < p.H ? sample_of(p, v) : -1;
    m.pos = p.pos[m.o];
    m.slot = p.slot[m.o];
  }
  return m;
}

// Part 1, after QKV: one warp per (non-rejected row, head): the QKV shares'
// sum, scaled by the row's 1/rms (pre-norm), RoPE on q and k, q of the sample
// rows, k and v at the row's cache slot.  Lane l rotates the pairs (i, i + hd/2)
// for i = l and l + 32 (hd <= 128).
PE_DEV void stage_rope(const DecParams& p, int n_rows, const RopeMeta& first) {
  const int lane = threadIdx.x & 31;
  const int ew = (threadIdx.x >> 5) - 2;
  const int heads = p.H + 2 * p.G;
  const int half = p.hd / 2;
  const int nc = (p.d + kChunk - 1) / kChunk;
  for (int u = blockIdx.x * 4 + ew; u < n_rows * heads; u += gridDim.x * 4) {
    const int v = u / heads, hh = u - v * heads;
    const bool pre = u == first.u;
    const int o = pre ? first.o : p.valid_rows[v];
    const float share = p.post_norm ? 0.f : ss_share(p.ss, v, nc);
    int f[4];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int i = lane + 32 * q;
      f[2 * q] = i < half ? hh * p.hd + i : -1;
      f[2 * q + 1] = i < half ? hh * p.hd + i + half : -1;
    }
    float x[4];
    sum_parts<4, 8>(p.g[1], 0, v, f, x);
    const int s = pre ? first.s : (hh < p.H ? sample_of(p, v) : -1);
    const int64_t pos = pre ? first.pos : p.pos[o];
    const int64_t slot = pre ? first.slot : p.slot[o];
    const float sc = p.post_norm ? 1.f : inv_rms(share, p.d, p.eps);
    const bool slot_ok = slot >= 0 && slot < static_cast<int64_t>(p.num_blocks) * p.bs;
    if (!slot_ok && slot != PE_PADDING_SLOT_ID && lane == 0 && hh == 0)
      set_status(p.status, PE_ST_BLOCK_RANGE);
    const int64_t blk = slot_ok ? slot / p.bs : 0, off = slot_ok ? slot % p.bs : 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int i = lane + 32 * q;
      if (i >= half) continue;
      const float x1 = sc * x[2 * q], x2 = sc * x[2 * q + 1];
      if (hh >= p.H + p.G) {  // v: no rotation
        if (slot_ok) {
          bf16* vc = p.v_cache + ((blk * p.G + (hh - p.H - p.G)) * p.bs + off) * p.hd;
          vc[i] = __float2bfloat16_rn(x1);
          vc[i + half] = __float2bfloat16_rn(x2);
        }
        continue;
      }
      float sn, cs;
      rope_cos_sin(pos, first.turn[q], cs, sn);
      const float y1 = x1 * cs - x2 * sn;
      const float y2 = x2 * cs + x1 * sn;
      if (hh < p.H) {
        if (s >= 0) {
          bf16* qd = p.q_s + (static_cast<size_t>(s) * p.H + hh) * p.hd;
          qd[i] = __float2bfloat16_rn(y1);
          qd[i + half] = __float2bfloat16_rn(y2);
        }
      } else if (slot_ok) {
        bf16* kc = p.k_cache + ((blk * p.G + (hh - p.H)) * p.bs + off) * p.hd;
        kc[i] = __float2bfloat16_rn(y1);
        kc[i + half] = __float2bfloat16_rn(y2);
      }
    }
  }
}

// Part 2, after O: r = x_s + the O shares' sum; the MLP operand r * gamma_post
// as a bf16 pair; per-chunk sums of squares of r.
PE_DEV void stage_after_o(const DecParams& p, float* red) {
  const int nc = (p.d + kChunk - 1) / kChunk;
  const int cg = chunks_per_unit(p.rows_cap, nc);
  const int ngr = (nc + cg - 1) / cg;
  for (int u = blockIdx.x; u < p.rows_cap * ngr; u += gridDim.x) {
    const int s = u / ngr, c0 = (u - s * ngr) * cg;
    int f[kMaxCG];
    unit_features(c0, cg, p.d, f);
    float xs[kMaxCG], x[kMaxCG];
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i)
      xs[i] = f[i] >= 0 ? p.x_s[static_cast<size_t>(s) * p.d + f[i]] : 0.f;
    sum_parts<kMaxCG, 16>(p.g[0], 0, s, f, x);
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i) {
      float rv = 0.f;
      if (f[i] >= 0) {
        const size_t k = static_cast<size_t>(s) * p.d + f[i];
        rv = xs[i] + x[i];
        p.r[k] = rv;
        store_pair(p.op_hi, p.op_lo, k, rv * __bfloat162float(p.gamma_a[f[i]]));
      }
      x[i] = rv * rv;
    }
    sum128(x, red);
    if (threadIdx.x == 64)
#pragma unroll
      for (int i = 0; i < kMaxCG; ++i)
        if (i < cg && c0 + i < nc) p.ss[s * 64 + c0 + i] = x[i];
  }
}

// Part 2, after gate/up: h = silu(g) * u with g, u the shares' sums scaled by
// the row's 1/rms (the MLP input is RMSNorm(r) * gamma_post), as a bf16 pair.
PE_DEV void stage_swiglu(const DecParams& p) {
  const int nc = (p.inter + kChunk - 1) / kChunk;
  const int ncd = (p.d + kChunk - 1) / kChunk;
  const int cg = chunks_per_unit(p.rows_cap, nc);
  const int ngr = (nc + cg - 1) / cg;
  const int up = p.g[1].splits * kDecodeRows * p.g[1].M;  // matrix 1 as a feature offset
  for (int u = blockIdx.x; u < p.rows_cap * ngr; u += gridDim.x) {
    const int s = u / ngr, c0 = (u - s * ngr) * cg;
    const float share = ss_share(p.ss, s, ncd);
    int f[kMaxCG], fgu[2 * kMaxCG];
    unit_features(c0, cg, p.inter, f);
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i) {
      fgu[i] = f[i];
      fgu[kMaxCG + i] = f[i] >= 0 ? f[i] + up : -1;
    }
    float x[2 * kMaxCG];
    sum_parts<2 * kMaxCG, 8>(p.g[1], 0, s, fgu, x);
    const float sc = inv_rms(share, p.d, p.eps);
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i) {
      if (f[i] < 0) continue;
      const float gv = sc * x[i];
      const float uv = sc * x[kMaxCG + i];
      store_pair(p.h_hi, p.h_lo, static_cast<size_t>(s) * p.inter + f[i],
                 gv / (1.0f + expf(-gv)) * uv);
    }
  }
}

// Part 2, after down: y = residual + the down shares' sum (residual: r
// pre-norm; RMSNorm(r) * gamma_post post-norm); per-chunk sums of squares of y.
PE_DEV void stage_after_down(const DecParams& p, float* red) {
  const int nc = (p.d + kChunk - 1) / kChunk;
  const int cg = chunks_per_unit(p.rows_cap, nc);
  const int ngr = (nc + cg - 1) / cg;
  for (int u = blockIdx.x; u < p.rows_cap * ngr; u += gridDim.x) {
    const int s = u / ngr, c0 = (u - s * ngr) * cg;
    const float share = p.post_norm ? ss_share(p.ss, s, nc) : 0.f;
    int f[kMaxCG];
    unit_features(c0, cg, p.d, f);
    float rr[kMaxCG], x[kMaxCG];
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i)
      rr[i] = f[i] >= 0 ? p.r[static_cast<size_t>(s) * p.d + f[i]] : 0.f;
    sum_parts<kMaxCG, 16>(p.g[2], 0, s, f, x);
    const float sc = p.post_norm ? inv_rms(share, p.d, p.eps) : 1.f;
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i) {
      float yv = 0.f;
      if (f[i] >= 0) {
        const size_t k = static_cast<size_t>(s) * p.d + f[i];
        const float res = p.post_norm ? sc * rr[i] * __bfloat162float(p.gamma_a[f[i]]) : rr[i];
        yv = res + x[i];
        p.y[k] = yv;
      }
      x[i] = yv * yv;
    }
    sum128(x, red);
    if (threadIdx.x == 64)
#pragma unroll
      for (int i = 0; i < kMaxCG; ++i)
        if (i < cg && c0 + i < nc) p.ss2[s * 64 + c0 + i] = x[i];
  }
}

// Part 2, last: z = RMSNorm(y) * gamma_final (bf16) and the hidden state handed
// on (y pre-norm, the normalised value post-norm).
PE_DEV void stage_final(const DecParams& p) {
  const int nc = (p.d + kChunk - 1) / kChunk;
  const int cg = chunks_per_unit(p.rows_cap, nc);
  const int ngr = (nc + cg - 1) / cg;
  for (int u = blockIdx.x; u < p.rows_cap * ngr; u += gridDim.x) {
    const int s = u / ngr, c0 = (u - s * ngr) * cg;
    const float share = ss_share(p.ss2, s, nc);
    int f[kMaxCG];
    unit_features(c0, cg, p.d, f);
    float yv[kMaxCG];
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i)
      yv[i] = f[i] >= 0 ? p.y[static_cast<size_t>(s) * p.d + f[i]] : 0.f;
    const float sc = inv_rms(share, p.d, p.eps);
#pragma unroll
    for (int i = 0; i < kMaxCG; ++i) {
      if (f[i] < 0) continue;
      const size_t k = static_cast<size_t>(s) * p.d + f[i];
      const float zf = yv[i] * sc * __bfloat162float(p.gamma_b[f[i]]);
      p.z[k] = __float2bfloat16_rn(zf);
      if (p.hidden_out) p.hidden_out[k] = p.post_norm ? zf : yv[i];
    }
  }
}

// ---------------------------------------------------------------- the kernel

// PART 1: fc, [after fc], QKV, [RoPE].  PART 2: O, [after O], gate/up,
// [SwiGLU], down, [after down], [final].  The barrier word after GEMM stage
// `gs` (its partial tiles stored) and after each elementwise stage.
template <int PART>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_layer_kernel(const __grid_constant__ DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kSlots], empty_bar[kSlots], tfull_bar, tempty_bar,
      final_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, ok_sh;
  __shared__ float red_sh[4 * kMaxCG];
  __shared__ uint32_t epoch_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int wbase = PART == 1 ? BW_PART1 : BW_PART2;
  const int wepoch = PART == 1 ? BW_EPOCH1 : BW_EPOCH2;
  // barrier word that releases GEMM stage gs's token operand (-1: the kernel before)
  auto ready_word = [&](int gs) { return gs == 0 ? -1 : wbase + 2 * gs - 1; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tfull_bar, 1);
    mbar_init(&tempty_bar, 128);
    mbar_init(&final_bar, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_sh;
  volatile int* abort_flag = &abort_sh;

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int slot = 0;
      uint32_t phase = 0, armed = 0u, armed_parity = 0u;
      uint32_t target = 0;
      bool have_target = false, ok = true;
      for (int gs = 0; gs < p.n_gemm && ok; ++gs) {
        const DecGemm& g = p.g[gs];
        Item it;
        const bool mine = item_of(g, blockIdx.x, it);
        const CUtensorMap* mA = &p.mapA[gs][mine ? it.mat : 0];
        const uint32_t bytes = kABytes + kBBytes * (g.bpair ? 2u : 1u);
        int pre_slot[kSlots];
        int pre = 0;
        if (mine) {
          prefetch_tmap(mA);
          // the weight boxes of the first ring stages go out before the wait
          const int want = min(it.kb1 - it.kb0, kSlots);
          for (int j = 0; j < want; ++j) {
            if (!mbar_wait(&empty_bar[slot], phase ^ 1u, abort_flag)) {
              ok = false;
              if (!*abort_flag) abort_all(p, PART, 10 + gs);
              break;
            }
            mbar_arrive_expect_tx(&full_bar[slot], bytes);
            int cx, cy;
            weight_box(g, it.m, it.kb0 + j, cx, cy);
            tma_load_2d(smem + static_cast<size_t>(slot) * kSlotBytes, mA, &full_bar[slot], cx, cy,
                        pol_w);
            armed |= 1u << slot;
            armed_parity = (armed_parity & ~(1u << slot)) | (phase << slot);
            pre_slot[pre++] = slot;
            if (++slot == kSlots) {
              slot = 0;
              phase ^= 1u;
            }
          }
        }
        // the token operand: written by the kernel before, or the stage before
        if (!have_target) {
          pdl_wait();
          target = (ld_acquire(p.bar + wepoch) + 1u) * gridDim.x;
          have_target = true;
        }
        if (ok && ready_word(gs) >= 0) {
          if (!grid_wait(p, ready_word(gs), target)) {
            ok = false;
            abort_all(p, PART, 1 + gs, ready_word(gs), target);
          } else {
            fence_proxy_async_global();
          }
        }
        if (!ok) {
          // the stages armed above still get their token boxes, so they complete
          for (int j = 0; j < pre && mine; ++j) {
            uint8_t* sb = smem + static_cast<size_t>(pre_slot[j]) * kSlotBytes + kABytes;
            tma_load_2d(sb, &p.mapB[gs][0], &full_bar[pre_slot[j]], (it.kb0 + j) * kBK, 0, pol_x);
            if (g.bpair)
              tma_load_2d(sb + kBBytes, &p.mapB[gs][1], &full_bar[pre_slot[j]], (it.kb0 + j) * kBK,
                          0, pol_x);
          }
          break;
        }
        if (!mine) continue;
        for (int j = 0; j < pre; ++j) {
          uint8_t* sb = smem + static_cast<size_t>(pre_slot[j]) * kSlotBytes + kABytes;
          tma_load_2d(sb, &p.mapB[gs][0], &full_bar[pre_slot[j]], (it.kb0 + j) * kBK, 0, pol_x);
          if (g.bpair)
            tma_load_2d(sb + kBBytes, &p.mapB[gs][1], &full_bar[pre_slot[j]], (it.kb0 + j) * kBK, 0,
                        pol_x);
        }
        for (int kb = it.kb0 + pre; kb < it.kb1; ++kb) {
          if (!mbar_wait(&empty_bar[slot], phase ^ 1u, abort_flag)) {
            ok = false;
            if (!*abort_flag) abort_all(p, PART, 20 + gs);
            break;
          }
          mbar_arrive_expect_tx(&full_bar[slot], bytes);
          uint8_t* sa = smem + static_cast<size_t>(slot) * kSlotBytes;
          int cx, cy;
          weight_box(g, it.m, kb, cx, cy);
          tma_load_2d(sa, mA, &full_bar[slot], cx, cy, pol_w);
          tma_load_2d(sa + kABytes, &p.mapB[gs][0], &full_bar[slot], kb * kBK, 0, pol_x);
          if (g.bpair) tma_load_2d(sa + kABytes + kBBytes, &p.mapB[gs][1], &full_bar[slot], kb * kBK, 0, pol_x);
          armed |= 1u << slot;
          armed_parity = (armed_parity & ~(1u << slot)) | (phase << slot);
          if (++slot == kSlots) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) abort_sh = 1;
      if (*abort_flag) {
        // copies already in flight land before the CTA's shared memory goes away
        for (int s = 0; s < kSlots; ++s)
          if (armed & (1u << s)) {
            int dummy = 0;
            mbar_wait(&full_bar[s], (armed_parity >> s) & 1u, &dummy);
          }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, kDecodeRows);
      int slot = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int gs = 0; gs < p.n_gemm && ok && !*abort_flag; ++gs) {
        const DecGemm& g = p.g[gs];
        Item it;
        if (!item_of(g, blockIdx.x, it)) continue;
        if (!mbar_wait(&tempty_bar, acc_phase ^ 1u, abort_flag)) {
          ok = false;
          if (!*abort_flag) abort_all(p, PART, 30 + gs);
          break;
        }
        tc_fence_after();
        for (int kb = it.kb0; kb < it.kb1; ++kb) {
          if (!mbar_wait(&full_bar[slot], phase, abort_flag)) {
            ok = false;
            if (!*abort_flag) abort_all(p, PART, 40 + gs);
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + static_cast<size_t>(slot) * kSlotBytes);
          const uint64_t adesc = sw128_kmajor_desc(sa);
          const uint64_t bdesc = sw128_kmajor_desc(sa + kABytes);
          const uint64_t b2desc = sw128_kmajor_desc(sa + kABytes + kBBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t acc = (kb > it.kb0 || kk > 0) ? 1u : 0u;
            umma_bf16(tmem_base, adesc + 2 * kk, bdesc + 2 * kk, idesc, acc);
            if (g.bpair) umma_bf16(tmem_base, adesc + 2 * kk, b2desc + 2 * kk, idesc, 1u);
          }
          umma_commit(&empty_bar[slot]);
          if (++slot == kSlots) {
            slot = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull_bar);
        acc_phase ^= 1u;
      }
      if (!ok) abort_sh = 1;
      umma_commit(&final_bar);
      int dummy = 0;
      mbar_wait(&final_bar, 0, &dummy);
    }
  } else {
    // ---------------- warps 2-5: partial tiles and the elementwise stages
    const int q = warp & 3;
    const int fl = q * 32 + lane;
    const int j = threadIdx.x - 64;
    pdl_wait();
    if (j == 0) epoch_sh = (ld_acquire(p.bar + wepoch) + 1u) * gridDim.x;
    named_bar_sync(1, 128);
    const uint32_t target = epoch_sh;
    int n_rows = p.rows_cap;
    if (p.n_rows_dev) n_rows = min(max(*p.n_rows_dev, 0), p.rows_cap);
    uint32_t acc_phase = 0;
    bool ok = true;
    // every CTA arrives at every barrier word, in order, once
    auto gemm_epilogue = [&](int gs) {
      const DecGemm& g = p.g[gs];
      Item it;
      if (item_of(g, blockIdx.x, it)) {
        const bool got = mbar_wait(&tfull_bar, acc_phase, abort_flag);
        if (j == 0) ok_sh = 1;
        named_bar_sync(1, 128);
        if (!got) {
          ok_sh = 0;
          if (j == 0 && !*abort_flag) abort_all(p, PART, 50 + gs);
        }
        named_bar_sync(1, 128);
        if (!ok_sh) return false;
        acc_phase ^= 1u;
        tc_fence_after();
        float v[16];
        tmem_ld16(tmem_base + (static_cast<uint32_t>(q * 32) << 16), v);
        tc_fence_before();
        mbar_arrive(&tempty_bar);
        const int f = it.m * kBM + fl;
        if (f < g.M) {
          float* out = g.out + (static_cast<size_t>(it.mat) * g.splits + it.ks) * kDecodeRows * g.M + f;
#pragma unroll
          for (int t = 0; t < kDecodeRows; ++t)
            if (t < n_rows) out[static_cast<size_t>(t) * g.M] = v[t];
        }
      }
      return true;
    };
    auto barrier = [&](int w, bool wait_next) {
      // arrive at w; then (wait_next) wait for every CTA's arrival at w
      named_bar_sync(1, 128);
      if (j == 0) {
        grid_arrive(p, w);
        ok_sh = wait_next ? (grid_wait(p, w, target) ? 1 : 0) : 1;
        if (!ok_sh) abort_all(p, PART, 60, w, target);
      }
      named_bar_sync(1, 128);
      return ok_sh != 0;
    };
    if (PART == 1) {
      // the row metadata of this CTA's first units, read while fc streams
      const RopeMeta rmeta = rope_meta(p, n_rows);
      int s_first = -1;
      {
        const int nc = (p.d + kChunk - 1) / kChunk;
        const int cg = chunks_per_unit(n_rows, nc);
        const int ngr = (nc + cg - 1) / cg;
        if (static_cast<int>(blockIdx.x) < n_rows * ngr) s_first = sample_of(p, blockIdx.x / ngr);
      }
      ok = gemm_epilogue(0) && barrier(wbase + 0, true);
      if (ok) stage_after_fc(p, n_rows, red_sh, s_first);
      ok = ok && barrier(wbase + 1, false);
      ok = ok && gemm_epilogue(1) && barrier(wbase + 2, true);
      if (ok) stage_rope(p, n_rows, rmeta);
    } else {
      ok = gemm_epilogue(0) && barrier(wbase + 0, true);
      if (ok) stage_after_o(p, red_sh);
      ok = ok && barrier(wbase + 1, false);
      ok = ok && gemm_epilogue(1) && barrier(wbase + 2, true);
      if (ok) stage_swiglu(p);
      ok = ok && barrier(wbase + 3, false);
      ok = ok && gemm_epilogue(2) && barrier(wbase + 4, true);
      if (ok) stage_after_down(p, red_sh);
      ok = ok && barrier(wbase + 5, true);
      if (ok) stage_final(p);
    }
    if (!ok && j == 0) abort_sh = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  // the last CTA to finish counts the launch (every CTA has read the count by now)
  if (threadIdx.x == 64) {
    const int wdone = PART == 1 ? BW_PART1 + 3 : BW_PART2 + 6;
    __threadfence();
    const uint32_t prev = atomicAdd(p.bar + wdone, 1u);
    if (prev + 1u == epoch_sh) atomicAdd(p.bar + wepoch, 1u);
  }
}

}  // namespace

// ---------------------------------------------------------------- host

size_t decode_scratch_bytes(int d, int qkv, int inter, int num_sms) {
  // partial tiles: the largest projection's shares over every CTA of the grid
  const size_t grid = static_cast<size_t>(num_sms) * kCtasPerSm;
  const size_t rows = kDecodeRows;
  const int widest = std::max(std::max(d, qkv), inter);
  const size_t parts = grid * rows * kBM * sizeof(float) + rows * widest * sizeof(float) * 2;
  auto a256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  return a256(parts) +                                          // partial tiles
         2 * a256(rows * std::max(d, inter) * 2) +              // operand pair
         2 * a256(rows * inter * 2) +                           // SwiGLU pair
         2 * a256(rows * d * sizeof(float)) +                   // r, y
         2 * a256(rows * 64 * sizeof(float));                   // sums of squares
}

bool decode_layer_fits(int d, int qkv, int inter, int num_sms) {
  const int grid = num_sms * kCtasPerSm;
  auto tiles = [](int m) { return (m + kBM - 1) / kBM; };
  // every projection's weight tiles fit the grid; a row's chunk sums fit 64 slots
  return num_sms > 0 && tiles(d) <= grid && tiles(qkv) <= grid && 2 * tiles(inter) <= grid &&
         (d + kChunk - 1) / kChunk <= 64;
}

// Split a projection [M][K] (n_mats matrices) so that every CTA of the grid
// has at most one item.
static DecGemm plan_dec_gemm(int M, int K, int n_mats, int bpair, int grid, float* out) {
  DecGemm g{};
  g.M = M;
  g.K = K;
  g.n_mats = n_mats;
  g.bpair = bpair;
  g.m_tiles = (M + kBM - 1) / kBM;
  g.num_kb = (K + kBK - 1) / kBK;
  int s = std::max(1, grid / (n_mats * g.m_tiles));
  s = std::min(s, g.num_kb);
  g.kbps = (g.num_kb + s - 1) / s;
  g.splits = (g.num_kb + g.kbps - 1) / g.kbps;
  g.items = n_mats * g.m_tiles * g.splits;
  g.out = out;
  return g;
}

int launch_decode_layer(const DecodeLaunch& L, int part, cudaStream_t st) {
  const int grid = L.num_sms * kCtasPerSm;
  DecParams p;
  std::memset(&p, 0, sizeof(p));
  const int Hd = L.H * L.hd;
  const int QKV = (L.H + 2 * L.G) * L.hd;
  auto a256 = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  char* base = static_cast<char*>(L.scratch);
  const size_t rows = kDecodeRows;
  const int widest = std::max(std::max(L.d, QKV), L.inter);
  size_t off = 0;
  float* part_buf = reinterpret_cast<float*>(base + off);
  off += a256(static_cast<size_t>(grid) * rows * kBM * sizeof(float) +
              rows * widest * sizeof(float) * 2);
  bf16* op_hi = reinterpret_cast<bf16*>(base + off);
  off += a256(rows * std::max(L.d, L.inter) * 2);
  bf16* op_lo = reinterpret_cast<bf16*>(base + off);
  off += a256(rows * std::max(L.d, L.inter) * 2);
  bf16* h_hi = reinterpret_cast<bf16*>(base + off);
  off += a256(rows * L.inter * 2);
  bf16* h_lo = reinterpret_cast<bf16*>(base + off);
  off += a256(rows * L.inter * 2);
  float* r = reinterpret_cast<float*>(base + off);
  off += a256(rows * L.d * sizeof(float));
  float* y = reinterpret_cast<float*>(base + off);
  off += a256(rows * L.d * sizeof(float));
  float* ss = reinterpret_cast<float*>(base + off);
  off += a256(rows * 64 * sizeof(float));
  float* ss2 = reinterpret_cast<float*>(base + off);

  p.d = L.d;
  p.H = L.H;
  p.G = L.G;
  p.hd = L.hd;
  p.inter = L.inter;
  p.K = L.K;
  p.B = L.B;
  p.bs = L.bs;
  p.num_blocks = L.num_blocks;
  p.post_norm = L.post_norm;
  p.eps = L.eps;
  p.x_s = L.x_s;
  p.op_hi = op_hi;
  p.op_lo = op_lo;
  p.h_hi = h_hi;
  p.h_lo = h_lo;
  p.r = r;
  p.y = y;
  p.ss = ss;
  p.ss2 = ss2;
  p.bar = L.bar;
  p.status = L.status;
  std::memcpy(p.rope_turn, L.rope_turn, sizeof(p.rope_turn));
  auto map_x = [&](CUtensorMap* m, const void* X, int rows_cap, int cols) {
    return encode_tmap_bf16(m, X, static_cast<uint64_t>(rows_cap), static_cast<uint64_t>(cols),
                            kDecodeRows);
  };
  bool ok = true;
  if (part == 1) {
    p.rows_cap = L.T_out;
    p.n_rows_dev = L.n_valid;
    p.valid_rows = L.valid_rows;
    p.valid_qsl = L.valid_qsl;
    p.pos = L.pos;
    p.slot = L.slot;
    p.gamma_a = static_cast<const bf16*>(L.gamma_in);
    p.q_s = static_cast<bf16*>(L.q_s);
    p.k_cache = static_cast<bf16*>(L.k_cache);
    p.v_cache = static_cast<bf16*>(L.v_cache);
    p.n_gemm = 2;
    p.g[0] = plan_dec_gemm(L.d, 4 * L.d, 1, 0, grid, part_buf);
    p.g[1] = plan_dec_gemm(QKV, L.d, 1, 1, grid, part_buf);
    p.mapA[0][0] = *L.m_fc;
    p.mapA[1][0] = *L.m_qkv;
    ok = map_x(&p.mapB[0][0], L.A, L.T_out, 4 * L.d) && map_x(&p.mapB[1][0], op_hi, L.T_out, L.d) &&
         map_x(&p.mapB[1][1], op_lo, L.T_out, L.d);
    p.mapB[0][1] = p.mapB[0][0];
  } else {
    const int NS = L.B * L.K;
    p.rows_cap = NS;
    p.gamma_a = static_cast<const bf16*>(L.gamma_post);
    p.gamma_b = static_cast<const bf16*>(L.gamma_final);
    p.z = static_cast<bf16*>(L.z);
    p.hidden_out = L.hidden_out;
    p.n_gemm = 3;
    p.g[0] = plan_dec_gemm(L.d, Hd, 1, 0, grid, part_buf);
    p.g[1] = plan_dec_gemm(L.inter, L.d, 2, 1, grid, part_buf);
    p.g[2] = plan_dec_gemm(L.d, L.inter, 1, 1, grid, part_buf);
    p.mapA[0][0] = *L.m_o;
    p.mapA[1][0] = *L.m_gate;
    p.mapA[1][1] = *L.m_up;
    p.mapA[2][0] = *L.m_down;
    ok = map_x(&p.mapB[0][0], L.attn, NS, Hd) && map_x(&p.mapB[1][0], op_hi, NS, L.d) &&
         map_x(&p.mapB[1][1], op_lo, NS, L.d) && map_x(&p.mapB[2][0], h_hi, NS, L.inter) &&
         map_x(&p.mapB[2][1], h_lo, NS, L.inter);
    p.mapB[0][1] = p.mapB[0][0];
  }
  if (!ok) return PE_ERR_CUDA;
  auto kern = part == 1 ? decode_layer_kernel<1> : decode_layer_kernel<2>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) != cudaSuccess)
    return PE_ERR_CUDA;

  return launch_pdl(kern, dim3(grid), dim3(kThreads), kSmemBytes, st, p) == cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}

}  // namespace pe
