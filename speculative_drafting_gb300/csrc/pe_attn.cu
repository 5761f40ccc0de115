// Paged attention of the K draft queries of each request over its whole
// context plus the earlier draft positions ("P-EAGLE: parallel speculative
// decoding in vLLM", Parallel drafting: all positions pass through the layer at
// once; draft position k sees every cache position up to its own).
//
// bf16: one CTA per (request, KV head, key split).  Its query tile is the K
// sample rows x the H/G query heads that share the KV head (GQA).  A producer
// warp streams the KV blocks with TMA (one block-table lookup per 16 keys) into
// a 3-chunk ring; compute warps own 16 query rows and half of every 64-key
// chunk; S = Q K^T and O += P V run on warp-level bf16 mma.sync with fp32
// accumulators and an online softmax in the exp2 domain (P enters the second
// product as a hi + lo bf16 pair).  Each split leaves an unnormalised partial
// (flash-decoding style).  While the splits of a (request, KV head) fit one
// thread-block cluster they merge there, through distributed shared memory;
// otherwise the partials go to global memory and a combine kernel merges them.
//
// fp32: one CTA per (sample row, query head), SIMT dot products, online softmax.
//
// Optional per-head sink logits (the GPT-oss attention, "Attention Drift",
// section 3: a learned bias logit in each head's softmax denominator) enter
// where the partials are normalised: the sink joins the running maximum and adds
// its exponential to the denominator, with a zero value row.
#include <algorithm>
#include <cmath>

#include "pe_common.cuh"
#include "pe_prep.h"

namespace pe {

constexpr int kKC = 64;               // keys per chunk
constexpr int kStages = 3;            // KV chunks in flight per CTA
constexpr int kMaxComputeWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 128;       // key splits per (request, KV head)
constexpr long kMaxSplitKeys = 2048;  // keys per split, at most
// Cluster mode: the splits of one (request, KV head) are one thread-block
// cluster (non-portable size up to 16) and merge in distributed shared memory.
// Chosen while the whole grid is one wave (two CTAs per SM) and its splits stay
// at most kClusterSplitKeys keys long, or at most a quarter longer than the
// splits the global-memory merge would use.  With several waves a cluster's
// CTAs would hold their SMs while waiting for the cluster's slowest split
// (measured at B=64: +163 us, at B=32 with 32K contexts: +102 us).
constexpr int kMaxAttnCluster = 16;
constexpr long kClusterSplitKeys = 1024;

// Thread roles of the bf16 attention CTA: compute warps 0..cw-1 (row warp
// w % rw, key group w / rw), then one producer warp.
struct AttnShape {
  int rw;  // warps over the query rows (16 rows each)
  int kg;  // key groups: each handles 64 / kg keys of every chunk
  int cw;  // compute warps = rw * kg
};

__host__ __device__ inline AttnShape attn_shape(int rows) {
  AttnShape s;
  s.rw = (rows + 15) / 16;
  s.kg = s.rw <= kMaxComputeWarps / 2 ? 2 : 1;
  s.cw = s.rw * s.kg;
  return s;
}

// 2^x by the hardware approximation (ex2.approx.ftz: results below the normal
// range flush to 0, weights far below the rounding of any sum they join).
PE_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One CTA per (key split, KV head, request).  The producer warp walks the
// split's 64-key chunks: per 16-key group it looks the block up once and loads
// the K and V rows of this KV head with TMA (128-byte swizzle, 64 elements of
// the head dim per box) into a ring of kStages chunks.  Each compute warp owns
// 16 query rows and one key group; S = Q K^T and O += P V run on mma.sync with
// fp32 accumulators and an online softmax in the exp2 domain; P enters P V as a
// hi + lo bf16 pair.  At the end the key groups' states merge in shared memory
// and the CTA writes unnormalised partials for the combine kernel.
// MINB = 2 (hd = 64): registers capped so that two CTAs share an SM, for grids
// of several waves (one CTA's 3-chunk ring does not keep an SM's share of DRAM
// busy; measured at B=64: step 1756 -> 1570 us).  A grid of one wave keeps the
// uncapped registers (no spills).  hd = 128 fits two CTAs by shared memory.
template <int HD, int KG, int MINB>
__global__ void __launch_bounds__(32 * (kMaxComputeWarps + 1), MINB)
    attn_tma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const AttnArgs a) {
  constexpr int HALVES = HD / 64;        // 128-byte swizzle atoms per key row
  constexpr int GROUP_BYTES = 16 * 128;  // one box: 16 keys x 64 dims
  constexpr int TILE = kKC * HD * 2;     // one K (or V) chunk
  constexpr int STAGE = 2 * TILE;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ uint32_t mask_sh[kStages];
  __shared__ int abort_sh;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int HG = a.H / a.G;
  const int rows = a.K * HG;
  const AttnShape sh = attn_shape(rows);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int n_compute = sh.cw * 32;

  // stale shared memory must be finite: a masked key still multiplies its V row by 0
  for (int i = threadIdx.x; i < kStages * STAGE / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], sh.cw);
    }
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == sh.cw && lane == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  pdl_trigger();
  pdl_wait();
  fence_proxy_async();  // the zeroed ring is visible to the TMA writes that follow
  __syncthreads();

  // this CTA's unit: (split, KV head, request) from the grid, or entry
  // blockIdx.x of the longest-first order (attn_order_kernel); past its end the
  // CTA has nothing to do
  int split = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
  if (a.order) {
    const int n = a.order[0].x;
    const int idx = static_cast<int>(blockIdx.x);
    if (n >= 0) {
      if (idx >= n) return;
      const int2 e = a.order[1 + idx];
      r = e.x;
      split = e.y / a.G;
      g = e.y - split * a.G;
    } else {
      // split-major by index (batches too large to order)
      const int BG = a.B * a.G;
      split = idx / BG;
      r = (idx - split * BG) / a.G;
      g = idx - split * BG - r * a.G;
    }
  }

  int L = a.seq_len[r];
  const int Lmax = a.max_blocks * a.bs;
  if (L > Lmax || L < a.k_min) {
    if (threadIdx.x == 0) set_status(a.status, PE_ST_BLOCK_RANGE);
    L = min(max(L, 0), Lmax);
  }
  const int P0 = L - a.K;  // position of the first draft query (the NTP row)
  const int t0 = split * a.split_len;
  const int t1 = min(L, t0 + a.split_len);
  // a split past the request's keys: nothing to write, the combine stops
  // before it (a cluster's CTAs all take part in its merge)
  if (!a.cluster && split > 0 && t0 >= L) return;
  const int n_chunks = t1 > t0 ? (t1 - t0 + kKC - 1) / kKC : 0;
  const size_t n_samp = static_cast<size_t>(a.B) * a.K;
  volatile int* abort_flag = &abort_sh;

  if (warp == sh.cw) {
    // ---------------- producer warp: its lanes look up the KV rows of 32
    // 16-key groups (8 chunks) at once; lane 0 issues the loads
    int stage = 0;
    uint32_t phase = 0;
    bool go = true;
    for (int cb = 0; cb < n_chunks && go; cb += 8) {
      int rowv = -1;  // this lane's group: cache row of its first key, -1 = none
      {
        const int t = t0 + (cb * 4 + lane) * 16;
        if (t < t1) {
          const int blk = a.block_table[static_cast<size_t>(r) * a.max_blocks + t / a.bs];
          if (blk < 0 || blk >= a.num_blocks)
            set_status(a.status, PE_ST_BLOCK_RANGE);
          else
            rowv = (blk * a.G + g) * a.bs + t % a.bs;
        }
      }
      const int c_end = min(n_chunks, cb + 8);
      for (int c = cb; c < c_end; ++c) {
        int row[4];
        uint32_t mask = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          row[q] = __shfl_sync(0xffffffffu, rowv, (c - cb) * 4 + q);
          if (row[q] >= 0) mask |= 1u << q;
        }
        int ok = 1;
        if (lane == 0) {
          if (*abort_flag || !mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
            abort_sh = 1;
            set_status(a.status, PE_ST_TIMEOUT);
            ok = 0;
          } else {
            mask_sh[stage] = mask;
            mbar_arrive_expect_tx(&full_bar[stage],
                                  static_cast<uint32_t>(__popc(mask)) * 2u * HALVES * GROUP_BYTES);
            uint8_t* kd = ring + stage * STAGE;
            uint8_t* vd = kd + TILE;
            for (int q = 0; q < 4; ++q) {
              if (!(mask & (1u << q))) continue;
              for (int hh = 0; hh < HALVES; ++hh) {
                const int off = hh * (kKC * 128) + q * GROUP_BYTES;
                tma_load_2d(kd + off, &kmap, &full_bar[stage], hh * 64, row[q],
                            policy_evict_first());
                tma_load_2d(vd + off, &vmap, &full_bar[stage], hh * 64, row[q],
                            policy_evict_first());
              }
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          go = false;
          break;
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ---------------- compute warps
    const int rw = warp % sh.rw, kgi = warp / sh.rw;
    constexpr int KEYS = kKC / KG;  // keys of each chunk this warp handles (64 or 32)
    constexpr int NT = KEYS / 8;    // 8-key n-tiles
    const int kofs = kgi * KEYS;
    const int ra = rw * 16 + gq, rb = ra + 8;
    auto row_sample = [&](int rr) { return static_cast<size_t>(r) * a.K + rr / HG; };
    auto row_head = [&](int rr) { return g * HG + rr % HG; };
    uint32_t qf[HD / 16][4];
    {
      const bf16* q = static_cast<const bf16*>(a.q);
      const bf16* qa = ra < rows ? q + (row_sample(ra) * a.H + row_head(ra)) * HD : nullptr;
      const bf16* qb = rb < rows ? q + (row_sample(rb) * a.H + row_head(rb)) * HD : nullptr;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
        const int c0 = ks * 16 + tq * 2;
        qf[ks][0] = qa ? *reinterpret_cast<const uint32_t*>(qa + c0) : 0u;
        qf[ks][1] = qb ? *reinterpret_cast<const uint32_t*>(qb + c0) : 0u;
        qf[ks][2] = qa ? *reinterpret_cast<const uint32_t*>(qa + c0 + 8) : 0u;
        qf[ks][3] = qb ? *reinterpret_cast<const uint32_t*>(qb + c0 + 8) : 0u;
      }
    }
    const int lim_a = P0 + (ra < rows ? ra / HG : 0);
    const int lim_b = P0 + (rb < rows ? rb / HG : 0);
    float o[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    const float sc = kLog2e / sqrtf(static_cast<float>(HD));
    // shared-memory address of 16-byte unit ch (0 .. HD/8-1) of chunk key kk
    auto kv_addr = [&](uint32_t base, int kk, int ch) {
      return base + (ch >> 3) * (kKC * 128) + kk * 128 + (((ch & 7) ^ (kk & 7)) << 4);
    };
    int stage = 0;
    uint32_t phase = 0;
    for (int c = 0; c < n_chunks; ++c) {
      if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
        abort_sh = 1;
        set_status(a.status, PE_ST_TIMEOUT);
        break;
      }
      const uint32_t mask = mask_sh[stage];
      const uint32_t kb = smem_u32(ring + stage * STAGE);
      const uint32_t vb = kb + TILE;
      // S = Q K^T over this warp's keys: KEYS/8 n-tiles of 8 keys
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
          const int mat = lane >> 3;
          const int kk = kofs + nt * 8 + (mat >> 1) * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kv_addr(kb, kk, ks * 2 + (mat & 1)), b0, b1, b2, b3);
          mma_bf16_16816(s[nt], qf[ks], b0, b1);
          mma_bf16_16816(s[nt + 1], qf[ks], b2, b3);
        }
      }
      // mask (range, invalid blocks, causal limit), online softmax
      const int kbase = t0 + c * kKC + kofs;
      // this warp's keys of the chunk are all in range, in valid blocks and at or
      // before position P0, which every query row sees: no per-key mask (the
      // same for the whole warp)
      constexpr uint32_t kGroupBits = (1u << (KEYS / 16)) - 1u;
      const bool interior = kbase + KEYS <= t1 && kbase + KEYS - 1 <= P0 &&
                            ((mask >> (kofs >> 4)) & kGroupBits) == kGroupBits;
      float mx_a = -INFINITY, mx_b = -INFINITY;
      if (interior) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            s[nt][e] *= sc;
            s[nt][2 + e] *= sc;
            mx_a = fmaxf(mx_a, s[nt][e]);
            mx_b = fmaxf(mx_b, s[nt][2 + e]);
          }
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = kbase + nt * 8 + tq * 2 + e;
            const bool ok = t < t1 && ((mask >> ((kofs + nt * 8) >> 4)) & 1u);
            s[nt][e] = (ok && t <= lim_a) ? s[nt][e] * sc : -INFINITY;
            s[nt][2 + e] = (ok && t <= lim_b) ? s[nt][2 + e] * sc : -INFINITY;
            mx_a = fmaxf(mx_a, s[nt][e]);
            mx_b = fmaxf(mx_b, s[nt][2 + e]);
          }
        }
      }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float al_a = (mn_a == -INFINITY) ? 1.f : ex2_approx(m_a - mn_a);
      const float al_b = (mn_b == -INFINITY) ? 1.f : ex2_approx(m_b - mn_b);
      m_a = mn_a;
      m_b = mn_b;
      float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[nt][e] = (mn_a == -INFINITY) ? 0.f : ex2_approx(s[nt][e] - mn_a);
          s[nt][2 + e] = (mn_b == -INFINITY) ? 0.f : ex2_approx(s[nt][2 + e] - mn_b);
          ps_a += s[nt][e];
          ps_b += s[nt][2 + e];
        }
      }
      l_a = l_a * al_a + ps_a;
      l_b = l_b * al_b + ps_b;
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) {
        o[i][0] *= al_a;
        o[i][1] *= al_a;
        o[i][2] *= al_b;
        o[i][3] *= al_b;
      }
      // O += P V over this warp's keys, 16 keys per k-step
#pragma unroll
      for (int kk = 0; kk < NT / 2; ++kk) {
        uint32_t ph[4], pl[4];
        split_bf16x2(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
        split_bf16x2(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
        split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
        split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
        if constexpr (HD == 64) {
          // all V fragments of the 16 keys first, then the high parts into every
          // accumulator, then the low parts: an accumulator's two updates are
          // eight MMAs apart instead of back to back
          uint32_t bv[HD / 8][2];
#pragma unroll
          for (int nd = 0; nd < HD / 8; nd += 2) {
            const int mat = lane >> 3;
            const int key = kofs + kk * 16 + (mat & 1) * 8 + (lane & 7);
            ldmatrix_x4_trans(kv_addr(vb, key, nd + (mat >> 1)), bv[nd][0], bv[nd][1],
                              bv[nd + 1][0], bv[nd + 1][1]);
          }
#pragma unroll
          for (int nd = 0; nd < HD / 8; ++nd) mma_bf16_16816(o[nd], ph, bv[nd][0], bv[nd][1]);
#pragma unroll
          for (int nd = 0; nd < HD / 8; ++nd) mma_bf16_16816(o[nd], pl, bv[nd][0], bv[nd][1]);
        } else {
#pragma unroll
          for (int nd = 0; nd < HD / 8; nd += 2) {
            const int mat = lane >> 3;
            const int key = kofs + kk * 16 + (mat & 1) * 8 + (lane & 7);
            uint32_t b0, b1, b2, b3;
            ldmatrix_x4_trans(kv_addr(vb, key, nd + (mat >> 1)), b0, b1, b2, b3);
            mma_bf16_16816(o[nd], ph, b0, b1);
            mma_bf16_16816(o[nd + 1], ph, b2, b3);
            mma_bf16_16816(o[nd], pl, b0, b1);
            mma_bf16_16816(o[nd + 1], pl, b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[stage]);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    // merge the key groups through the (now idle) ring: groups 1..KG-1 park their
    // state in regions 0..KG-2 ([row][HD] each, then (m, l) per row), group 0
    // merges; the merged partial then takes region 0's place
    constexpr int NREG = KG > 1 ? KG - 1 : 1;
    const int rows_pad = sh.rw * 16;
    float* mo = reinterpret_cast<float*>(ring);
    float* mml = mo + static_cast<size_t>(NREG) * rows_pad * HD;
    named_bar_sync(1, n_compute);
    if (KG > 1 && kgi >= 1) {
      float* po = mo + static_cast<size_t>(kgi - 1) * rows_pad * HD;
      float* pml = mml + static_cast<size_t>(kgi - 1) * rows_pad * 2;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int rl = rw * 16 + gq + hf * 8;
#pragma unroll
        for (int nd = 0; nd < HD / 8; ++nd) {
          const int d = nd * 8 + tq * 2;
          po[rl * HD + d] = o[nd][hf * 2];
          po[rl * HD + d + 1] = o[nd][hf * 2 + 1];
        }
        if (tq == 0) {
          pml[rl * 2] = hf ? m_b : m_a;
          pml[rl * 2 + 1] = hf ? l_b : l_a;
        }
      }
    }
    named_bar_sync(1, n_compute);
    if (kgi == 0) {
      // merged (m, l) of rows ra, rb (all four lanes of a row read the parked
      // group-1 values before any lane overwrites them below)
      float mh[2], lh[2], w0h[2], wgh[2][NREG];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float m = hf ? m_b : m_a, l = hf ? l_b : l_a;
        float w0 = 1.f;
        const int rl = rw * 16 + gq + hf * 8;
#pragma unroll
        for (int g2 = 0; g2 < NREG; ++g2) wgh[hf][g2] = 0.f;
        if (KG > 1) {
          float M = m;
#pragma unroll
          for (int g2 = 0; g2 < KG - 1; ++g2) M = fmaxf(M, mml[(g2 * rows_pad + rl) * 2]);
          w0 = (m == -INFINITY) ? 0.f : exp2f(m - M);
          l *= w0;
#pragma unroll
          for (int g2 = 0; g2 < KG - 1; ++g2) {
            const float mg = mml[(g2 * rows_pad + rl) * 2];
            const float wg = (mg == -INFINITY) ? 0.f : exp2f(mg - M);
            l += mml[(g2 * rows_pad + rl) * 2 + 1] * wg;
            wgh[hf][g2] = wg;
          }
          m = M;
        }
        mh[hf] = m;
        lh[hf] = l;
        w0h[hf] = w0;
      }
      __syncwarp();
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int rr = hf ? rb : ra;
        const int rl = rw * 16 + gq + hf * 8;
        // cluster: this split's partial replaces the parked values in place
        // (each element is read and written by the same lane); else global
        float* po = mo + rl * HD;
        float* pml = mml + rl * 2;
        if (!a.cluster) {
          if (rr >= rows) continue;
          const size_t idx =
              (static_cast<size_t>(split) * n_samp + row_sample(rr)) * a.H + row_head(rr);
          po = a.part_o + idx * HD;
          pml = a.part_ml + idx * 2;
        }
#pragma unroll
        for (int nd = 0; nd < HD / 8; ++nd) {
          const int d = nd * 8 + tq * 2;
          float v0 = o[nd][hf * 2] * w0h[hf], v1 = o[nd][hf * 2 + 1] * w0h[hf];
#pragma unroll
          for (int g2 = 0; g2 < KG - 1; ++g2) {
            const float* pg = mo + static_cast<size_t>(g2) * rows_pad * HD + rl * HD;
            v0 += pg[d] * wgh[hf][g2];
            v1 += pg[d + 1] * wgh[hf][g2];
          }
          *reinterpret_cast<float2*>(po + d) = make_float2(v0, v1);
        }
        if (tq == 0) {
          pml[0] = mh[hf];
          pml[1] = lh[hf];
        }
      }
    }
  }
  // the producer may still be waiting for an empty slot only after an abort
  __syncthreads();
  if (!a.cluster) return;

  // ---------------- merge of the splits inside the cluster
  // Every split's partial sits at the start of its ring: o [row][HD] (fp32,
  // unnormalised), then (m, l) per row.  CTA `rank` merges rows rank, rank + S,
  // ...: out = sum_j 2^(m_j - M) o_j / (sum_j 2^(m_j - M) l_j + 2^(sink - M)), where
  // the optional sink term has a zero value row and M also covers it.
  cluster_sync_all();
  {
    const int S = static_cast<int>(gridDim.x);
    const int rank = static_cast<int>(cluster_ctarank());
    const int nw = static_cast<int>(blockDim.x >> 5);
    const uint32_t o_base = smem_u32(ring);
    constexpr int NREG_C = KG > 1 ? KG - 1 : 1;
    const uint32_t ml_base = o_base + static_cast<uint32_t>(NREG_C * sh.rw * 16 * HD * 4);
    constexpr int DPL = HD / 32;  // dims per lane
    for (int i = warp;; i += nw) {
      const int rr = rank + i * S;
      if (rr >= rows) break;
      float mj = -INFINITY, lj = 0.f;
      if (lane < S) {
        mj = ld_dsmem_f32(ml_base + static_cast<uint32_t>(rr * 2) * 4u, lane);
        lj = ld_dsmem_f32(ml_base + static_cast<uint32_t>(rr * 2 + 1) * 4u, lane);
      }
      const int head = g * HG + rr % HG;
      // a sink logit (exp2 domain) joins the maximum and the denominator
      const float sk = a.sink ? a.sink[head] * kLog2e : -INFINITY;
      const float M = fmaxf(warp_max(mj), sk);
      const float wj = (mj == -INFINITY) ? 0.f : exp2f(mj - M);
      const float den = warp_sum(wj * lj) + (sk == -INFINITY ? 0.f : exp2f(sk - M));
      const float inv = den > 0.f ? 1.f / den : 0.f;
      float acc[DPL];
#pragma unroll
      for (int q = 0; q < DPL; ++q) acc[q] = 0.f;
      for (int j0 = 0; j0 < S; j0 += 4) {
        // four splits' loads in flight before their adds (in split order)
        float v[4][DPL];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int q = 0; q < DPL; ++q)
            v[u][q] = (j0 + u < S) ? ld_dsmem_f32(o_base + static_cast<uint32_t>(rr * HD + lane + 32 * q) * 4u,
                                                  static_cast<uint32_t>(j0 + u))
                                   : 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = __shfl_sync(0xffffffffu, wj, (j0 + u) & 31);
          if (j0 + u < S)
#pragma unroll
            for (int q = 0; q < DPL; ++q) acc[q] += w * v[u][q];
        }
      }
      const size_t samp = static_cast<size_t>(r) * a.K + rr / HG;
      bf16* out = static_cast<bf16*>(a.out) + (samp * a.H + head) * HD;
#pragma unroll
      for (int q = 0; q < DPL; ++q) out[lane + 32 * q] = __float2bfloat16_rn(acc[q] * inv);
    }
  }
  // no CTA leaves while another may still read its shared memory
  cluster_sync_all();
}

// out[s][h*hd + d] = sum_j 2^(m_j - M) o_j[d] / (sum_j 2^(m_j - M) l_j + 2^(sink_h - M))
// (the sink term only with sink logits) over the splits j that hold keys of the request (j * split_len < L; the CTAs of the
// others return at once and leave no partial).  One warp per (sample row,
// query head): each lane owns hd/32 consecutive dimensions; the splits' loads
// are independent, their sum runs in split order.
template <typename T, int HD>
__global__ void __launch_bounds__(128) attn_combine_kernel(const AttnArgs a) {
  constexpr int V = HD / 32;
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t n_sh = static_cast<size_t>(a.B) * a.K * a.H;
  const size_t sh = static_cast<size_t>(blockIdx.x) * 4 + warp;  // (sample, head)
  if (sh >= n_sh) return;
  const int r = static_cast<int>(sh / (static_cast<size_t>(a.K) * a.H));
  const int L = min(max(a.seq_len[r], 0), a.max_blocks * a.bs);
  const int n = max(1, min(a.n_splits, (L + a.split_len - 1) / a.split_len));
  auto ml = [&](int j) { return a.part_ml + (static_cast<size_t>(j) * n_sh + sh) * 2; };
  float M = -INFINITY;
  for (int j = lane; j < n; j += 32) M = fmaxf(M, ml(j)[0]);
  // a sink logit (exp2 domain) joins the maximum and the denominator
  const float sk = a.sink ? a.sink[sh % a.H] * kLog2e : -INFINITY;
  M = fmaxf(warp_max(M), sk);
  float den = 0.f;
  for (int j = lane; j < n; j += 32) {
    const float m = ml(j)[0];
    den += (m == -INFINITY ? 0.f : exp2f(m - M)) * ml(j)[1];
  }
  den = warp_sum(den) + (sk == -INFINITY ? 0.f : exp2f(sk - M));
  const float inv = den > 0.f ? 1.f / den : 0.f;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < n; j0 += 32) {
    float w = 0.f;
    if (j0 + lane < n) {
      const float m = ml(j0 + lane)[0];
      w = m == -INFINITY ? 0.f : exp2f(m - M);
    }
    const int cnt = min(32, n - j0);
#pragma unroll 4
    for (int u = 0; u < cnt; ++u) {
      const float wu = __shfl_sync(0xffffffffu, w, u);
      const float* po = a.part_o + (static_cast<size_t>(j0 + u) * n_sh + sh) * HD + lane * V;
      if constexpr (V == 4) {
        const float4 x = *reinterpret_cast<const float4*>(po);
        acc[0] += wu * x.x;
        acc[1] += wu * x.y;
        acc[2] += wu * x.z;
        acc[3] += wu * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(po);
        acc[0] += wu * x.x;
        acc[1] += wu * x.y;
      }
    }
  }
  T* out = static_cast<T*>(a.out) + sh * HD + lane * V;
  if constexpr (sizeof(T) == 2) {
    // the lane's V = 2 or 4 bf16 outputs with one 4- or 8-byte store
    uint32_t w[V / 2];
#pragma unroll
    for (int i = 0; i < V / 2; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
      w[i] = *reinterpret_cast<const uint32_t*>(&h);
    }
    if constexpr (V == 2)
      *reinterpret_cast<uint32_t*>(out) = w[0];
    else
      *reinterpret_cast<uint2*>(out) = make_uint2(w[0], w[1]);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) out[i] = Elem<T>::from_f(acc[i] * inv);
  }
}

// fp32: one CTA (4 warps) per (sample row, query head)
__global__ void __launch_bounds__(128) attn_f32_kernel(const AttnArgs a) {
  __shared__ float wm[4], wl[4], wacc[4][128];
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, h = blockIdx.y;
  const int r = s / a.K, k = s % a.K;
  const int g = h / (a.H / a.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int L = a.seq_len[r];
  const int Lmax = a.max_blocks * a.bs;
  if (L > Lmax || L < a.k_min) {
    if (threadIdx.x == 0) set_status(a.status, PE_ST_BLOCK_RANGE);
    L = min(max(L, 0), Lmax);
  }
  const int lim = min(L - a.K + k, L - 1);  // inclusive
  const float* q = static_cast<const float*>(a.q) + (static_cast<size_t>(s) * a.H + h) * a.hd;
  float qv[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 4; ++i) qv[i] = (lane + 32 * i < a.hd) ? q[lane + 32 * i] : 0.f;
  const float scale = 1.0f / sqrtf(static_cast<float>(a.hd));
  float m = -INFINITY, l = 0.f;
  const float* kc = static_cast<const float*>(a.k_cache);
  const float* vc = static_cast<const float*>(a.v_cache);
  for (int t = warp; t <= lim; t += 4) {
    const int blk = a.block_table[static_cast<size_t>(r) * a.max_blocks + t / a.bs];
    if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) set_status(a.status, PE_ST_BLOCK_RANGE);
      continue;
    }
    const size_t base = ((static_cast<size_t>(blk) * a.G + g) * a.bs + t % a.bs) * a.hd;
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (lane + 32 * i < a.hd) dot = fmaf(qv[i], kc[base + lane + 32 * i], dot);
    const float sc = warp_sum(dot) * scale;
    const float mn = fmaxf(m, sc);
    const float al = expf(m - mn);
    const float p = expf(sc - mn);
    l = l * al + p;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (lane + 32 * i < a.hd) acc[i] = acc[i] * al + p * vc[base + lane + 32 * i];
    m = mn;
  }
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = l;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (lane + 32 * i < a.hd) wacc[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  // a sink logit joins the maximum and the denominator (its value row is zero)
  const float sk = a.sink ? a.sink[h] : -INFINITY;
  float M = sk;
  for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w]);
  float den = sk == -INFINITY ? 0.f : expf(sk - M);
  for (int w = 0; w < 4; ++w)
    if (wm[w] != -INFINITY) den += expf(wm[w] - M) * wl[w];
  for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
    float num = 0.f;
    for (int w = 0; w < 4; ++w)
      if (wm[w] != -INFINITY) num += expf(wm[w] - M) * wacc[w][d];
    static_cast<float*>(a.out)[(static_cast<size_t>(s) * a.H + h) * a.hd + d] =
        den > 0.f ? num / den : 0.f;
  }
}

// Key splits per (request, KV head): enough CTAs for two per SM, and no split
// longer than kMaxSplitKeys keys (long contexts of a large batch would
// otherwise leave a few CTAs streaming the longest contexts alone).
int attention_split_count(int B, int G, int max_blocks, int bs, int num_sms) {
  const long Lmax = static_cast<long>(max_blocks) * bs;
  const long chunks = std::max<long>(1, (Lmax + kKC - 1) / kKC);
  const long heads = std::max<long>(1, static_cast<long>(B) * G);
  long ns = (2L * std::max(num_sms, 1) + heads - 1) / heads;
  ns = std::max(ns, (Lmax + kMaxSplitKeys - 1) / kMaxSplitKeys);
  ns = std::max<long>(1, std::min(std::min(ns, chunks), static_cast<long>(kMaxSplits)));
  return static_cast<int>(ns);
}

void plan_attention(int B, int G, int K, int H, int hd, int max_blocks, int bs, int num_sms,
                    int& n_splits, int& split_len, int& cluster) {
  (void)K;
  (void)H;
  (void)hd;
  const long Lmax = static_cast<long>(max_blocks) * bs;
  const long chunks = std::max<long>(1, (Lmax + kKC - 1) / kKC);
  const long ns = attention_split_count(B, G, max_blocks, bs, num_sms);
  // as many splits as one cluster takes, if each stays short enough
  const long nc = std::min<long>(ns, kMaxAttnCluster);
  const long len_c = (chunks + nc - 1) / nc * kKC;
  const long len_g = (chunks + ns - 1) / ns * kKC;
  const long grid_c = static_cast<long>(B) * G * ((Lmax + len_c - 1) / len_c);
  if (grid_c <= 2L * num_sms && len_c <= std::max(kClusterSplitKeys, len_g + len_g / 4)) {
    cluster = 1;
    split_len = static_cast<int>(len_c);
  } else {
    cluster = 0;
    split_len = static_cast<int>(len_g);
  }
  n_splits = static_cast<int>((Lmax + split_len - 1) / split_len);
  if (n_splits < 1) n_splits = 1;
}

// The order in which a grid of several waves takes its units (split j, KV head
// g, request r), longest first: the hardware starts CTAs in index order as SMs
// free up, and the last units to start decide when the grid ends.  Every full
// split (split_len keys) comes first, in the grid's order (request, KV head,
// split); then each request's last,
// shorter split by its 64-key chunks, most first and in request order among
// equals; an empty context's first split last.  Splits past a request's keys
// are left out.  order[0].x = the number of entries (-1: more than kOrdMax
// requests, the grid takes its units split-major by index); order[1 + i] =
// (r, j G + g).  One warp.
constexpr int kOrdMax = 1024;
__global__ void __launch_bounds__(32) attn_order_kernel(const AttnArgs a, int2* order) {
  __shared__ int full_pre[kOrdMax + 1];  // full splits of the requests before r
  __shared__ int bstart[34];             // bucket offsets (33 buckets: 0..32 chunks)
  pdl_trigger();
  pdl_wait();  // the lengths come from the metadata kernel; the last grid has read order
  const int lane = threadIdx.x;
  if (a.B > kOrdMax) {
    if (lane == 0) order[0] = make_int2(-1, 0);
    return;
  }
  const int Lmax = a.max_blocks * a.bs;
  // -> the bucket of request r's last split (its chunks, 1..32; 0: an empty
  // context; -1: none), nf = its full splits
  auto req_class = [&](int r, int& nf) -> int {
    const int L = min(max(a.seq_len[r], 0), Lmax);
    nf = min(L / a.split_len, a.n_splits);
    const int rem = L - nf * a.split_len;
    if (rem > 0) return min((rem + kKC - 1) / kKC, 32);
    return L == 0 ? 0 : -1;
  };
  for (int i = lane; i < 34; i += 32) bstart[i] = 0;
  if (lane == 0) full_pre[0] = 0;
  __syncwarp();
  int base = 0;
  for (int r0 = 0; r0 < a.B; r0 += 32) {
    const int r = r0 + lane;
    int nf = 0, bk = -1;
    if (r < a.B) bk = req_class(r, nf);
    int incl = nf;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    if (r < a.B) full_pre[r + 1] = base + incl;
    if (bk >= 0) atomicAdd(&bstart[bk], 1);
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
  if (lane == 0) {
    int acc = 0;
    for (int bkt = 32; bkt >= 0; --bkt) {
      const int c = bstart[bkt];
      bstart[bkt] = acc;
      acc += c;
    }
    bstart[33] = acc;
  }
  __syncwarp();
  const int n_full = base * a.G;
  const int n_live = n_full + bstart[33] * a.G;
  // the full splits in the grid's own order (request, then KV head, then
  // split): entry u belongs to request r with G full_pre[r] <= u < G full_pre[r + 1]
  for (int u = lane; u < n_full; u += 32) {
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (full_pre[mid] * a.G <= u)
        lo = mid;
      else
        hi = mid;
    }
    const int nf = full_pre[lo + 1] - full_pre[lo];
    const int loc = u - full_pre[lo] * a.G;
    const int gg = loc / nf, j = loc - gg * nf;
    order[1 + u] = make_int2(lo, j * a.G + gg);
  }
  // the last splits: each request's place in its bucket, in request order
  for (int r0 = 0; r0 < a.B; r0 += 32) {
    const int r = r0 + lane;
    int nf = 0, bk = -1;
    if (r < a.B) bk = req_class(r, nf);
    const unsigned same = __match_any_sync(0xffffffffu, bk);
    const int s0 = bk >= 0 ? bstart[bk] : 0;
    __syncwarp();
    const unsigned below = same & ((1u << lane) - 1u);
    if (bk >= 0) {
      const int pos = s0 + __popc(below);
      const int j = min(nf, a.n_splits - 1);
      for (int gg = 0; gg < a.G; ++gg) order[1 + n_full + pos * a.G + gg] = make_int2(r, j * a.G + gg);
      if (below == 0) bstart[bk] = s0 + __popc(same);
    }
    __syncwarp();
  }
  if (lane == 0) order[0] = make_int2(n_live, 0);
}

size_t attention_scratch_bytes(int B, int K, int H, int hd, int n_splits) {
  const size_t sh = static_cast<size_t>(n_splits) * B * K * H;
  size_t o = sh * hd * sizeof(float);
  o = (o + 255) / 256 * 256;
  size_t ml = sh * 2 * sizeof(float);
  ml = (ml + 255) / 256 * 256;
  // the unit order: at most n_splits * B * H units (G <= H), plus the count
  size_t ord = (static_cast<size_t>(n_splits) * B * H + 1) * sizeof(int2);
  ord = (ord + 255) / 256 * 256;
  return o + ml + ord;
}

int launch_attention(const AttnArgs& a, int dtype, cudaStream_t st) {
  if (a.B <= 0) return PE_OK;
  if (dtype != PE_DTYPE_BF16) {
    return launch_pdl(attn_f32_kernel, dim3(a.B * a.K, a.H), dim3(128), 0, st, a) == cudaSuccess
               ? PE_OK
               : PE_ERR_CUDA;
  }
  const int rows = a.K * (a.H / a.G);
  const AttnShape sh = attn_shape(rows);
  const dim3 grid(a.n_splits, a.G, a.B);
  const size_t smem = static_cast<size_t>(kStages) * 2 * kKC * a.hd * 2 + 1024;
  // TMA views of the caches: rows = (block, KV head, offset), 64-element boxes
  // of 16 rows; a 16-key group never crosses a block (block size % 16 == 0)
  CUtensorMap kmap, vmap;
  const uint64_t nrows = static_cast<uint64_t>(a.num_blocks) * a.G * a.bs;
  if (!encode_tmap_bf16(&kmap, a.k_cache, nrows, a.hd, 16) ||
      !encode_tmap_bf16(&vmap, a.v_cache, nrows, a.hd, 16))
    return PE_ERR_CUDA;
  const int smem_max = kStages * 2 * kKC * 128 * 2 + 1024;
  const dim3 block(32 * (sh.cw + 1));
  void (*kern)(CUtensorMap, CUtensorMap, AttnArgs) = nullptr;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool waves = static_cast<long>(grid.x) * grid.y * grid.z > sms;
  const dim3 cgrid(static_cast<unsigned>((static_cast<size_t>(a.B) * a.K * a.H + 3) / 4));
  auto combine = [&](const AttnArgs& ag) {
    return launch_pdl(a.hd == 64 ? attn_combine_kernel<bf16, 64> : attn_combine_kernel<bf16, 128>,
                      cgrid, dim3(128), 0, st, ag) == cudaSuccess
               ? PE_OK
               : PE_ERR_CUDA;
  };
  if (a.hd == 64) {
    // the register-capped instance (two CTAs per SM) for several waves
    kern = sh.kg == 2 ? (waves ? attn_tma_kernel<64, 2, 2> : attn_tma_kernel<64, 2, 1>)
                      : (waves ? attn_tma_kernel<64, 1, 2> : attn_tma_kernel<64, 1, 1>);
  } else if (a.hd == 128) {
    kern = sh.kg == 2 ? attn_tma_kernel<128, 2, 1> : attn_tma_kernel<128, 1, 1>;
  } else {
    return PE_ERR_UNSUPPORTED;
  }
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
  cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                       cudaSharedmemCarveoutMaxShared);
  if (a.cluster) {
    // one cluster per (request, KV head): the splits merge in shared memory
    if (a.n_splits > kMaxAttnCluster) return PE_ERR_UNSUPPORTED;
    if (a.n_splits > 8)
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(a.n_splits);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int n_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&n_clusters, (void*)kern, &cfg) == cudaSuccess &&
        n_clusters > 0)
      return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, a) == cudaSuccess ? PE_OK : PE_ERR_CUDA;
    cudaGetLastError();
    // the SMs cannot hold such a cluster: the same splits through global memory
    // (the workspace holds partials for at least this many splits)
  }
  AttnArgs ag = a;
  ag.cluster = 0;
  ag.order = nullptr;
  dim3 g3 = grid;
  if (waves && a.hd == 64) {
    // several waves at head size 64: the units in the longest-first order, one
    // CTA per entry; the order sits after the partials (attention_scratch_bytes).
    // Head size 128 keeps the 3-D grid: there the order measured slower (Llama-8B
    // shape, 32 requests of 32K keys: 1337 -> 1396 us a step)
    const size_t sh = static_cast<size_t>(a.n_splits) * a.B * a.K * a.H;
    const size_t ml = (sh * 2 * sizeof(float) + 255) / 256 * 256;
    ag.order = reinterpret_cast<int2*>(reinterpret_cast<char*>(a.part_ml) + ml);
    if (launch_pdl(attn_order_kernel, dim3(1), dim3(32), 0, st, ag, ag.order) != cudaSuccess)
      return PE_ERR_CUDA;
    g3 = dim3(static_cast<unsigned>(static_cast<size_t>(a.n_splits) * a.G * a.B));
  }
  if (launch_pdl(kern, g3, block, smem, st, kmap, vmap, ag) != cudaSuccess) return PE_ERR_CUDA;
  return combine(ag);
}

}  // namespace pe
