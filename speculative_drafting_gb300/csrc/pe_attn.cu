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
#include <type_traits>

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

  const int split = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
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

// ---------------------------------------------------------------- tcgen05 attention (hd = 64)
// For hd = 64 and query tiles of at most 64 rows (K x H/G), both products run on
// the tensor cores (tcgen05) with fp32 accumulators in tensor memory:
//   S = Q K^T (M = 128, N = 64 keys, K = 64 dims): Q is read from tensor memory,
//             its rows 0..63 the query rows, rows 64..127 the same rows again;
//   O += P V  (M = 128, N = 64 dims, K = 64 keys): rows 0..63 of P hold the high
//             bf16 part of the softmax weights, rows 64..127 the low part (the
//             hi + lo pair, about 16 significant bits), so one MMA covers both
//             halves and a query row's output is O[r] + O[r + 64].
// The kernel is persistent: two CTAs per SM take work units (key split j, KV head
// g, request r) from a counter in global memory, longest first (the claim order
// below), and stream one unit's 64-key chunks after the other through the same
// pipeline, so the ring stays full across unit boundaries.  Each unit leaves the same partial as the
// mma.sync kernel's CTAs (unnormalised o, then m and l in the exp2 domain) for
// the combine kernel.  Warp 0 claims units and streams K and V with TMA (every
// ring stage carries its unit, its chunk index and its group mask); one thread
// of warp 1 issues the MMAs; each thread of warps 2..5 owns one TMEM lane R.
// Lanes r and r + 64 hold the same score row: both take its maximum over the
// chunk's 64 keys, each takes the exponentials of half the keys (lane r the first
// 32, lane r + 64 the last 32) and writes their hi and lo weights into the P
// tile.  O accumulates in tensor memory over a unit's chunks; a row's reference
// maximum moves only when a score exceeds it by more than kTcRescale (weights up
// to 2^kTcRescale), and then each of its two lanes rescales its O row in place
// between two P V products.  Q sits in tensor memory, double-buffered by unit:
// the next unit's rows are copied into a staging tile (cp.async) when a unit
// starts and moved into tensor memory after its first chunk.
constexpr int kTcStages = 4;
constexpr int kTcTile = kKC * 64 * 2;   // one K (or V) chunk: 64 keys x 64 dims bf16
constexpr int kTcStage = 2 * kTcTile;   // K then V
constexpr int kTcRowBytes = 128 * 128;  // 128 rows x 128 bytes: the P tile, the Q staging tile
constexpr int kTcSmem = kTcStages * kTcStage + 2 * kTcRowBytes + 1024;
constexpr uint32_t kTcTmemCols = 256;   // S0, S1, O: 64 fp32 columns each; Q0, Q1: 32 each
constexpr uint32_t kTcOCol = 128;
constexpr uint32_t kTcQCol = 192;       // Q (two bf16 per column), buffer b at + 32 b
constexpr int kTcRows = 64;             // query rows per unit, at most
constexpr int kTcUq = 4;                // ring of claimed unit ids
constexpr float kTcRescale = 8.f;
constexpr int kTcOrdMax = 1024;         // requests whose units are claimed longest first
// dynamic + static shared memory (the claim order, 8 bytes per request, and
// the rest) + the 1 KB the system reserves, twice per SM
static_assert(2 * (kTcSmem + 8 * kTcOrdMax + 2048) <= 228 * 1024, "two tcgen05 attention CTAs per SM");
static_assert(2 * kTcTmemCols <= 512, "two tcgen05 attention CTAs per SM (tensor memory)");
static_assert(kTcRows * 64 * 4 <= kTcRowBytes, "a unit's o rows fit the P tile");
static_assert(kTcQCol + 64 <= kTcTmemCols, "both Q buffers fit the tensor memory");

// Shared-memory descriptor of an MN-major bf16 tile with the 128-byte swizzle:
// 128-byte rows of 64 consecutive N elements, one row per K index, 8-row atoms
// of 1024 bytes.  A 64-wide N is one atom wide, so the only stride the MMA
// walks is the 1024 bytes between the atoms of 8 K rows; both offset fields
// hold it.
PE_DEV uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1024 >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// max(a, b, c) in one instruction
PE_DEV float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// D[tmem] (+)= A[tmem] * B[smem]^T, A read from tensor memory (one row per
// lane, two bf16 per 32-bit column, K-major), issued by one thread.
PE_DEV void umma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Has the phase of parity `parity` completed?  (No waiting.)
PE_DEV bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// N consecutive 32-bit columns of this thread's TMEM lane (32x32b shape, thread
// t of the warp reads or writes lane taddr.lane + t), waited for in the same
// statement so that no use of the registers can move above the wait.
PE_DEV void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
PE_DEV void tmem_st32(uint32_t taddr, const float* v) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;\n"
      :
      : "r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
PE_DEV void tmem_st64(uint32_t taddr, const float* v) {
  uint32_t r[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};\n\t"
      "tcgen05.wait::st.sync.aligned;\n"
      :
      : "r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]),
        "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]),
        "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]),
        "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]),
        "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}


// A work unit of the tcgen05 attention: key split j of request r, KV head g.
// Units are numbered split-major: u = (j B + r) G + g.
struct TcUnit {
  int r, g, j;
  int L;       // the request's keys (clamped to its block table)
  int t0, t1;  // the split's keys [t0, t1)
  int n;       // 64-key chunks
};

// A unit's fields as the producer hands them to the softmax warps:
// (u, r, g | j << 16, L); u = -1: no unit left.
PE_DEV TcUnit tc_unit_of(const AttnArgs& a, int4 e) {
  TcUnit x;
  x.r = e.y;
  x.g = e.z & 0xffff;
  x.j = e.z >> 16;
  x.L = e.w;
  x.t0 = x.j * a.split_len;
  x.t1 = min(x.L, x.t0 + a.split_len);
  x.n = x.t1 > x.t0 ? (x.t1 - x.t0 + kKC - 1) / kKC : 0;
  return x;
}

PE_DEV TcUnit tc_unit_jrg(const AttnArgs& a, int j, int r, int g) {
  TcUnit x;
  x.j = j;
  x.r = r;
  x.g = g;
  x.L = min(max(a.seq_len[r], 0), a.max_blocks * a.bs);
  x.t0 = x.j * a.split_len;
  x.t1 = min(x.L, x.t0 + a.split_len);
  x.n = x.t1 > x.t0 ? (x.t1 - x.t0 + kKC - 1) / kKC : 0;
  return x;
}

// Unit u in split-major order.
PE_DEV TcUnit tc_unit(const AttnArgs& a, int u) {
  const int BG = a.B * a.G;
  const int j = u / BG;
  const int rem = u - j * BG;
  return tc_unit_jrg(a, j, rem / a.G, rem % a.G);
}

__global__ void __launch_bounds__(192, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kTcStages], empty_bar[kTcStages];
  __shared__ __align__(8) uint64_t s_full[2], q_full[2], uq_full[kTcUq], uq_empty[kTcUq];
  __shared__ __align__(8) uint64_t p_full, o_done, x_full, x_empty, done_bar;
  __shared__ int4 meta_sh[kTcStages];  // per stage: unit (-1: end of the stream), chunk, chunks, group mask
  __shared__ int4 uq_sh[kTcUq];        // claimed units' fields, in this CTA's order (tc_unit_of)
  __shared__ float xl_sh[kTcRows];     // the low lanes' sums of weights, at a unit's end
  // the claim order (producer warp): full splits per request as a prefix, the
  // requests ordered by the chunks of their last split, and its bucket offsets
  __shared__ int ord_full[kTcOrdMax + 1];
  __shared__ int ord_part[kTcOrdMax];
  __shared__ int ord_start[34];
  __shared__ uint32_t tmem_sh;
  __shared__ int abort_sh;
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // P tile, [128 rows][64 keys] bf16, K-major with the 128-byte swizzle; at a
  // unit's end it carries the low lanes' O rows to the high lanes
  uint8_t* pbuf = ring + kTcStages * kTcStage;
  uint8_t* qst = pbuf + kTcRowBytes;  // the next unit's Q rows, [128][128 bytes], swizzled

  const int HG = a.H / a.G;
  const int rows = a.K * HG;
  const int U = a.n_splits * a.G * a.B;
  const int Lmax = a.max_blocks * a.bs;
  const size_t n_samp = static_cast<size_t>(a.B) * a.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // stale shared memory must be finite: a masked key still multiplies its V row by 0
  for (int i = threadIdx.x; i < kTcStages * kTcStage / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&q_full[b], 128);
    }
    for (int i = 0; i < kTcUq; ++i) {
      mbar_init(&uq_full[i], 1);
      mbar_init(&uq_empty[i], 128);
    }
    mbar_init(&p_full, 128);
    mbar_init(&o_done, 1);
    mbar_init(&x_full, kTcRows);
    mbar_init(&x_empty, kTcRows);
    mbar_init(&done_bar, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
  }
  // tensor memory before the next kernel may start: its CTAs then find this
  // grid's allocations in place and wait for them, never the other way round
  if (warp == 1) {
    tmem_alloc(&tmem_sh, kTcTmemCols);
    tmem_relinquish();
  }
  pdl_trigger();
  pdl_wait();
  fence_proxy_async();  // the zeroed ring is visible to the TMA writes that follow
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_sh;
  volatile int* abort_flag = &abort_sh;
  auto fail = [&]() {
    abort_sh = 1;
    set_status(a.status, PE_ST_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------- producer warp.  It claims each unit one ahead of the one
    // it streams (while the ring is full), reads the block ids of the next
    // 8-chunk window one window ahead (across unit boundaries too), and issues
    // the TMA loads of each chunk into the ring.
    constexpr int GROUP_BYTES = 16 * 128;  // one box: 16 keys x 64 dims
    constexpr int kPast = -0x7fffffff - 1;  // a group past the split's keys
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0u, armed_parity = 0u;  // per stage: ever filled / parity of its last fill
    bool go = true;
    // The claim order, longest units first (as dealt by a shared counter, the
    // last units decide when the grid ends): every split of split_len keys,
    // request-major, then each request's last, shorter split by its chunks,
    // most first and in request order among equals, an empty context's empty
    // split last.  Every CTA builds the same order from the request lengths.
    // Larger batches take the splits split-major.
    const bool lpt = a.B <= kTcOrdMax;
    int n_full = 0, n_live = 0;  // units of full splits; units with keys or an empty context
    // -> the bucket of request r's last split: its chunks (1..32), 0 for an
    // empty context, -1 for none; nf = its full splits
    auto req_class = [&](int r, int& nf) -> int {
      const int L = min(max(a.seq_len[r], 0), Lmax);
      nf = min(L / a.split_len, a.n_splits);
      const int rem = L - nf * a.split_len;
      if (rem > 0) return min((rem + kKC - 1) / kKC, 32);
      return L == 0 ? 0 : -1;
    };
    if (lpt) {
      for (int i = lane; i < 34; i += 32) ord_start[i] = 0;
      if (lane == 0) ord_full[0] = 0;
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
        if (r < a.B) ord_full[r + 1] = base + incl;
        if (bk >= 0) atomicAdd(&ord_start[bk], 1);
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncwarp();
      if (lane == 0) {
        int acc = 0;
        for (int bkt = 32; bkt >= 0; --bkt) {
          const int c = ord_start[bkt];
          ord_start[bkt] = acc;
          acc += c;
        }
        ord_start[33] = acc;
      }
      __syncwarp();
      n_full = base * a.G;
      n_live = n_full + ord_start[33] * a.G;
      // each request's place in its bucket, in request order
      for (int r0 = 0; r0 < a.B; r0 += 32) {
        const int r = r0 + lane;
        int nf = 0, bk = -1;
        if (r < a.B) bk = req_class(r, nf);
        const unsigned same = __match_any_sync(0xffffffffu, bk);
        const int s0 = bk >= 0 ? ord_start[bk] : 0;
        __syncwarp();
        const unsigned below = same & ((1u << lane) - 1u);
        if (bk >= 0) {
          ord_part[s0 + __popc(below)] = r;
          if (below == 0) ord_start[bk] = s0 + __popc(same);
        }
        __syncwarp();
      }
    }
    // the next unit with keys (x = -1: none left); an empty context's first
    // split leaves its empty partial here, and splits past a request's keys none
    auto claim = [&]() -> int4 {
      for (;;) {
        int u = 0;
        if (lane == 0) u = static_cast<int>(atomicAdd(a.sched, 1u));
        u = __shfl_sync(0xffffffffu, u, 0);
        TcUnit x;
        if (lpt) {
          if (u >= n_live) return make_int4(-1, 0, 0, 0);
          if (u < n_full) {
            // full split j of request r: ord_full[r] <= u / G < ord_full[r + 1]
            const int up = u / a.G;
            int lo = 0, hi = a.B;
            while (hi - lo > 1) {
              const int mid = (lo + hi) >> 1;
              if (ord_full[mid] <= up)
                lo = mid;
              else
                hi = mid;
            }
            x = tc_unit_jrg(a, up - ord_full[lo], lo, u - up * a.G);
          } else {
            const int v = u - n_full;
            const int pos = v / a.G;
            const int r = ord_part[pos];
            const int L = min(max(a.seq_len[r], 0), Lmax);
            x = tc_unit_jrg(a, min(L / a.split_len, a.n_splits - 1), r, v - pos * a.G);
          }
        } else {
          if (u >= U) return make_int4(-1, 0, 0, 0);
          x = tc_unit(a, u);
          if (x.j > 0 && x.t0 >= x.L) continue;
        }
        if (lane == 0) {
          const int Lr = a.seq_len[x.r];
          if (Lr > Lmax || Lr < a.k_min) set_status(a.status, PE_ST_BLOCK_RANGE);
        }
        if (x.n == 0) {
          for (int rr = 0; rr < rows; ++rr) {
            const size_t idx =
                (static_cast<size_t>(x.j) * n_samp + static_cast<size_t>(x.r) * a.K + rr / HG) * a.H +
                x.g * HG + rr % HG;
            a.part_o[idx * 64 + lane] = 0.f;
            a.part_o[idx * 64 + 32 + lane] = 0.f;
            if (lane == 0) {
              a.part_ml[idx * 2] = -INFINITY;
              a.part_ml[idx * 2 + 1] = 0.f;
            }
          }
          continue;
        }
        return make_int4(u, x.r, x.g | (x.j << 16), x.L);
      }
    };
    // unit number k of this CTA's sequence, for the softmax warps
    auto publish = [&](int k, int4 e) -> bool {
      const int sl = k % kTcUq;
      int ok = 1;
      if (lane == 0) {
        if (k >= kTcUq && !mbar_wait(&uq_empty[sl], (k / kTcUq - 1) & 1, abort_flag)) {
          ok = 0;
        } else {
          uq_sh[sl] = e;
          mbar_arrive(&uq_full[sl]);
        }
      }
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    // block id of this lane's 16-key group of window cbw of unit y (the load's
    // value is used one window later)
    auto load_blk = [&](const TcUnit& y, int cbw) -> int {
      const int t = y.t0 + (cbw * 4 + lane) * 16;
      return t < y.t1 ? a.block_table[static_cast<size_t>(y.r) * a.max_blocks + t / a.bs] : kPast;
    };
    // -> cache row of the group's first key, -1 = none
    auto to_row = [&](const TcUnit& y, int cbw, int blk) -> int {
      if (blk == kPast) return -1;
      if (blk < 0 || blk >= a.num_blocks) {
        set_status(a.status, PE_ST_BLOCK_RANGE);
        return -1;
      }
      const int t = y.t0 + (cbw * 4 + lane) * 16;
      return (blk * a.G + y.g) * a.bs + t % a.bs;
    };
    int4 ec = claim();  // the unit being streamed
    go = publish(0, ec);
    int4 en = make_int4(-1, 0, 0, 0);  // the one after it
    if (go && ec.x >= 0) {
      en = claim();
      go = publish(1, en);
    }
    int k = 0;
    TcUnit x = tc_unit_of(a, ec);
    int cb = 0;
    int blk = (go && ec.x >= 0) ? load_blk(x, 0) : kPast;
    while (go && ec.x >= 0) {
      // the next window: this unit's next 8 chunks, or the next unit's first
      const bool same = cb + 8 < x.n;
      const TcUnit xn = same ? x : tc_unit_of(a, en);
      const int cbn = same ? cb + 8 : 0;
      const int blk_next = (same || en.x >= 0) ? load_blk(xn, cbn) : kPast;
      const int rowv = to_row(x, cb, blk);
      const int c_end = min(x.n, cb + 8);
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
            ok = 0;
          } else {
            meta_sh[stage] = make_int4(ec.x, c, x.n, static_cast<int>(mask));
            mbar_arrive_expect_tx(&full_bar[stage], static_cast<uint32_t>(__popc(mask)) * 2u * GROUP_BYTES);
            uint8_t* kd = ring + stage * kTcStage;
            for (int q = 0; q < 4; ++q) {
              if (!(mask & (1u << q))) continue;
              tma_load_2d(kd + q * GROUP_BYTES, &kmap, &full_bar[stage], 0, row[q], policy_evict_first());
              tma_load_2d(kd + kTcTile + q * GROUP_BYTES, &vmap, &full_bar[stage], 0, row[q],
                          policy_evict_first());
            }
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          go = false;
          break;
        }
        if (++stage == kTcStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!go) break;
      if (same) {
        cb += 8;
      } else {
        // on to the next unit; the one after it is claimed now, with the ring full
        ++k;
        ec = en;
        x = xn;
        cb = 0;
        if (ec.x >= 0) {
          en = claim();
          if (!publish(k + 1, en)) {
            go = false;
            break;
          }
        }
      }
      blk = blk_next;
    }
    // the end of the stream: a stage without keys
    if (lane == 0) {
      if (go && mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
        meta_sh[stage] = make_int4(-1, 0, 0, 0);
        mbar_arrive(&full_bar[stage]);
      } else {
        fail();
        // let copies already in flight land before the CTA's shared memory goes away
        for (int s = 0; s < kTcStages; ++s)
          if (armed & (1u << s)) {
            int dummy = 0;
            mbar_wait(&full_bar[s], (armed_parity >> s) & 1u, &dummy);
          }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer.  Chunk c's S goes out as soon as its keys (and,
    // for a unit's first chunk, its Q) are there, if the softmax is done with the
    // S buffer (it has written P of chunk c - 2); P V of chunk c once P is
    // written.  The thread blocks in the barrier waits (no spinning beside the
    // softmax warps).
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, 64);
      const uint32_t idesc_o = idesc_bf16_f32(128, 64) | (1u << 16);  // B = V, MN-major
      const uint64_t pdesc = sw128_kmajor_desc(smem_u32(pbuf));
      int ns = 0;    // chunks whose S has been issued
      int kq = -1;   // unit of the Q those S products use
      bool end = false;
      // S of chunk ns if its inputs are there (block: wait for them); false
      // only for a wait that gave up
      auto try_s = [&](bool block) -> bool {
        const int stage = ns % kTcStages;
        const uint32_t par = (ns / kTcStages) & 1;
        if (block) {
          if (!mbar_wait(&full_bar[stage], par, abort_flag)) return false;
        } else if (!mbar_test(&full_bar[stage], par)) {
          return true;
        }
        const int4 md = meta_sh[stage];
        if (md.x < 0) {
          end = true;
          return true;
        }
        if (md.y == 0) {
          const int q = kq + 1;
          if (block) {
            if (!mbar_wait(&q_full[q & 1], (q >> 1) & 1, abort_flag)) return false;
          } else if (!mbar_test(&q_full[q & 1], (q >> 1) & 1)) {
            return true;
          }
          kq = q;
        }
        tc_fence_after();
        const uint64_t kdesc = sw128_kmajor_desc(smem_u32(ring + stage * kTcStage));
        // 16 dims per MMA: 8 columns of Q, 32 bytes along a K row
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ta(tmem + (ns & 1) * 64, tmem + kTcQCol + 32 * (kq & 1) + 8 * kk, kdesc + 2 * kk,
                       idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(&s_full[ns & 1]);
        ++ns;
        return true;
      };
      bool ok = try_s(true);
      for (int c = 0; ok && c < ns; ++c) {
        if (!end && ns == c + 1 && !(ok = try_s(false))) break;
        if (!mbar_wait(&p_full, c & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int stage = c % kTcStages;
        const int4 md = meta_sh[stage];
        const uint64_t vdesc = sw128_mnmajor_desc(smem_u32(ring + stage * kTcStage + kTcTile));
        // 16 keys per MMA: 32 bytes along a P row, 16 V rows of 128 bytes; a
        // unit's first chunk starts O afresh
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + kTcOCol, pdesc + 2 * kk, vdesc + 128 * kk, idesc_o, (md.y > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&o_done);
        umma_commit(&empty_bar[stage]);
        if (!end && ns == c + 1) ok = try_s(true);
      }
      if (!ok) fail();
      // every MMA done before the tensor memory is freed
      umma_commit(&done_bar);
      int dummy = 0;
      mbar_wait(&done_bar, 0, &dummy);
    }
    __syncwarp();
  } else {
    // ---------------- softmax warps: thread = TMEM lane R
    const int qd = warp & 3;
    const int R = qd * 32 + lane;
    const int qr = R & (kTcRows - 1);  // query row
    const int half = R >> 6;           // 0: high parts of P and O, keys 0..31; 1: low parts, keys 32..63
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(qd * 32) << 16);
    const int swz = qr & 7;
    const uint32_t off_hi = static_cast<uint32_t>((qr >> 3) * 1024 + swz * 128);  // P row qr
    const uint32_t off_lo = off_hi + 8 * 1024;                                   // P row qr + 64
    uint8_t* qst_row = qst + R * 128;
    const float sc = kLog2e / sqrtf(64.f);
    // this lane's row of Q for unit x (rows past the query tile are zero)
    auto q_src = [&](const TcUnit& x) -> const uint4* {
      return reinterpret_cast<const uint4*>(
          static_cast<const bf16*>(a.q) +
          ((static_cast<size_t>(x.r) * a.K + qr / HG) * a.H + x.g * HG + qr % HG) * 64);
    };
    auto q_to_tmem = [&](const uint4* v, int buf) {
      float qw[32];
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        qw[4 * ch] = __uint_as_float(v[ch].x);
        qw[4 * ch + 1] = __uint_as_float(v[ch].y);
        qw[4 * ch + 2] = __uint_as_float(v[ch].z);
        qw[4 * ch + 3] = __uint_as_float(v[ch].w);
      }
      tmem_st32(t_lane + kTcQCol + 32 * buf, qw);
      tc_fence_before();
      mbar_arrive(&q_full[buf]);
    };
    bool ok = true;
    int k = 0;  // this CTA's unit number
    {
      // unit 0's Q (its entry is released when the unit starts)
      const bool got = mbar_wait(&uq_full[0], 0, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        fail();
        ok = false;
      } else {
        const int4 e0 = uq_sh[0];
        if (e0.x >= 0) {
          uint4 v[8];
          const TcUnit x0 = tc_unit_of(a, e0);
          const uint4* src = q_src(x0);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) v[ch] = qr < rows ? src[ch] : make_uint4(0, 0, 0, 0);
          q_to_tmem(v, 0);
        }
      }
    }
    TcUnit x{};
    int P0 = 0, lim = 0;
    float m = -INFINITY, l = 0.f;
    bool q_pending = false, x_pending = false;
    int kx = 0;  // the unit whose pair exchange is pending
    for (int c = 0; ok; ++c) {
      const int stage = c % kTcStages;
      const bool got_f = mbar_wait(&full_bar[stage], (c / kTcStages) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, got_f)) {
        fail();
        break;
      }
      const int4 md = meta_sh[stage];
      if (md.x < 0) break;  // the end of the stream
      if (md.y == 0) {
        // unit k starts: its keys and causal limits (its entry was waited for
        // when unit k - 1 started); the next unit's Q rows go into the staging
        // tile while this unit's first chunk is processed
        x = tc_unit_of(a, uq_sh[k % kTcUq]);
        P0 = x.L - a.K;
        lim = P0 + (qr < rows ? qr / HG : 0);
        m = -INFINITY;
        l = 0.f;
        const int sl = (k + 1) % kTcUq;
        const bool got_u = mbar_wait(&uq_full[sl], ((k + 1) / kTcUq) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, got_u)) {
          fail();
          break;
        }
        const int4 en = uq_sh[sl];
        mbar_arrive(&uq_empty[k % kTcUq]);
        if (en.x >= 0) {
          const TcUnit xn = tc_unit_of(a, en);
          const uint4* src = qr < rows ? q_src(xn) : static_cast<const uint4*>(a.q);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            cp_async16(smem_u32(qst_row + ((ch ^ (R & 7)) << 4)), src + (qr < rows ? ch : 0), qr < rows);
          cp_async_commit();
          q_pending = true;
        }
      }
      const bool got_s = mbar_wait(&s_full[c & 1], (c >> 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, got_s)) {
        fail();
        break;
      }
      tc_fence_after();
      const uint32_t mask = static_cast<uint32_t>(md.w);
      const int kbase = x.t0 + md.y * kKC;
      // every key in range, in a valid block and at or before P0 (seen by all rows)
      const bool interior = kbase + kKC <= x.t1 && kbase + kKC - 1 <= P0 && mask == 0xFu;
      const uint32_t scol = static_cast<uint32_t>((c & 1) * 64);
      float sv[64];  // the chunk's 64 scores of this row
      tmem_ld64(t_lane + scol, sv);
      if (!interior) {
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int t = kbase + j;
          sv[j] = (t < x.t1 && ((mask >> (j >> 4)) & 1u) && t <= lim) ? sv[j] : -INFINITY;
        }
      }
      // the maximum of all 64: a tree of three-input maxima
      float mr;
      {
        float z[22], w[8];
#pragma unroll
        for (int i = 0; i < 21; ++i) z[i] = fmax3(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
        z[21] = sv[63];
#pragma unroll
        for (int i = 0; i < 7; ++i) w[i] = fmax3(z[3 * i], z[3 * i + 1], z[3 * i + 2]);
        w[7] = z[21];
        mr = fmax3(fmax3(w[0], w[1], w[2]), fmax3(w[3], w[4], w[5]), fmaxf(w[6], w[7]));
      }
      const float mx = mr * sc;  // in the exp2 domain (sc > 0)
      const bool move = mx > m + kTcRescale;
      const float mn = move ? mx : m;
      const float al = move ? ex2_approx(m - mn) : 1.f;
      // with no valid key so far every score of the chunk is -inf: any finite
      // reference gives the weights 0
      const float mref = (mn == -INFINITY) ? 0.f : mn;
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t hw[16], lw[16];
      // this lane's 32 keys (a constant offset into sv, so sv stays in registers)
      auto weights = [&](auto first) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const float p0 = ex2_approx(fmaf(sv[decltype(first)::value + j], sc, -mref));
          const float p1 = ex2_approx(fmaf(sv[decltype(first)::value + j + 1], sc, -mref));
          ps[(j >> 1) & 3] += p0 + p1;
          split_bf16x2(p0, p1, hw[j >> 1], lw[j >> 1]);
        }
      };
      if (half)
        weights(std::integral_constant<int, 32>{});
      else
        weights(std::integral_constant<int, 0>{});
      // the P tile is free once P V of chunk c - 1 has completed and (after a
      // unit's end) the high lanes have read the exchange; a moved reference
      // maximum then rescales O (within a unit)
      if (c >= 1) {
        const bool got_o = mbar_wait(&o_done, (c - 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, got_o)) {
          fail();
          break;
        }
        tc_fence_after();
      }
      if (x_pending) {
        const bool got_x = mbar_wait(&x_empty, kx & 1, abort_flag);
        if (!__all_sync(0xffffffffu, got_x)) {
          fail();
          break;
        }
        x_pending = false;
      }
      if (md.y > 0 && __any_sync(0xffffffffu, move)) {
        float ov[64];
        tmem_ld64(t_lane + kTcOCol, ov);
#pragma unroll
        for (int j = 0; j < 64; ++j) ov[j] *= al;
        tmem_st64(t_lane + kTcOCol, ov);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t col = static_cast<uint32_t>(((half * 4 + kk) ^ swz) << 4);
        *reinterpret_cast<uint4*>(pbuf + off_hi + col) =
            make_uint4(hw[4 * kk], hw[4 * kk + 1], hw[4 * kk + 2], hw[4 * kk + 3]);
        *reinterpret_cast<uint4*>(pbuf + off_lo + col) =
            make_uint4(lw[4 * kk], lw[4 * kk + 1], lw[4 * kk + 2], lw[4 * kk + 3]);
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(&p_full);
      l = l * al + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
      m = mn;
      if (q_pending) {
        // the next unit's Q into its tensor-memory buffer (its S products wait
        // for it; the buffer's previous unit has no S product left)
        cp_async_wait<0>();
        uint4 v[8];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) v[ch] = *reinterpret_cast<const uint4*>(qst_row + ((ch ^ (R & 7)) << 4));
        q_to_tmem(v, (k + 1) & 1);
        q_pending = false;
      }
      if (md.y == md.z - 1) {
        // unit k ends: its O rows, the two halves of the pair added, and its
        // partial for the combine kernel
        const bool got_o = mbar_wait(&o_done, c & 1, abort_flag);
        if (!__all_sync(0xffffffffu, got_o)) {
          fail();
          break;
        }
        tc_fence_after();
        float o[64];
        tmem_ld64(t_lane + kTcOCol, o);
        float* xo = reinterpret_cast<float*>(pbuf) + qr * 64;
        if (half) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            reinterpret_cast<float4*>(xo)[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          xl_sh[qr] = l;
          mbar_arrive(&x_full);
        } else {
          const bool got_x = mbar_wait(&x_full, k & 1, abort_flag);
          if (!__all_sync(0xffffffffu, got_x)) {
            fail();
            break;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float4 xv = reinterpret_cast<const float4*>(xo)[j];
            o[4 * j] += xv.x;
            o[4 * j + 1] += xv.y;
            o[4 * j + 2] += xv.z;
            o[4 * j + 3] += xv.w;
          }
          const float lt = l + xl_sh[qr];
          mbar_arrive(&x_empty);
          if (qr < rows) {
            const size_t idx =
                (static_cast<size_t>(x.j) * n_samp + static_cast<size_t>(x.r) * a.K + qr / HG) * a.H +
                x.g * HG + qr % HG;
            float4* dst = reinterpret_cast<float4*>(a.part_o + idx * 64);
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            a.part_ml[idx * 2] = m;
            a.part_ml[idx * 2 + 1] = lt;
          }
        }
        x_pending = true;
        kx = k;
        ++k;
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
  // the last CTA to finish leaves the unit counter at zero for the next launch
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
      a.sched[0] = 0u;
      a.sched[1] = 0u;
      __threadfence();
    }
  }
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

size_t attention_scratch_bytes(int B, int K, int H, int hd, int n_splits) {
  const size_t sh = static_cast<size_t>(n_splits) * B * K * H;
  size_t o = sh * hd * sizeof(float);
  o = (o + 255) / 256 * 256;
  size_t ml = sh * 2 * sizeof(float);
  ml = (ml + 255) / 256 * 256;
  return o + ml;
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
  if (a.hd == 64 && rows <= kTcRows && waves && !a.cluster && a.sched) {
    // several waves of units: the persistent tensor-core kernel, two CTAs per SM
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    const long units = static_cast<long>(a.n_splits) * a.G * a.B;
    const unsigned ctas = static_cast<unsigned>(std::min<long>(2L * sms, units));
    if (launch_pdl(attn_tc_kernel, dim3(ctas), dim3(192), kTcSmem, st, kmap, vmap, a) != cudaSuccess)
      return PE_ERR_CUDA;
    return combine(a);
  }
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
  if (launch_pdl(kern, grid, block, smem, st, kmap, vmap, ag) != cudaSuccess) return PE_ERR_CUDA;
  return combine(ag);
}

}  // namespace pe
