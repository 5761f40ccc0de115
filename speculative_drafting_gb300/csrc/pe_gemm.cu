// Drafter projections: D[t][f] = sum_k X[t][k] * W[f][k] with a fused epilogue.
//
// bf16: a persistent tcgen05 kernel.  The weight matrix is the MMA's M side
// (128 output features per tile) and the token rows are its N side (16..256
// per tile), so a decode-sized batch still fills the 128-row tensor-core tile
// and the weights stream through shared memory exactly once per N tile.  Warp 0
// issues TMA loads (128-byte swizzle, weights marked evict-first, tokens
// evict-last) into a ring of shared-memory stages; one thread of warp 1 issues
// tcgen05.mma into a TMEM accumulator; warps 2-5 read the accumulator with
// tcgen05.ld and run the epilogue.  Small-N projections split K across CTAs so
// every SM streams weights: the splits of a tile form a thread-block cluster
// and add their fp32 partial tiles through distributed shared memory, in rank
// order (deterministic), before the epilogue.
//
// fp32: a plain shared-memory-tiled SIMT kernel with the same epilogues (fp32
// FMA; TF32 would not meet a 1e-5 logit tolerance).
#include <algorithm>
#include <cstdio>
#include <map>
#include <mutex>

#include "pe_common.cuh"
#include "pe_internal.h"

namespace pe {

constexpr int kBM = 128;  // weight rows per tile (MMA M)
constexpr int kBK = 64;   // reduction elements per k-block: one 128-byte swizzle row
constexpr int kMaxStages = 12;
constexpr size_t kSmemBudget = 212 * 1024;  // dynamic shared memory for the stage ring
// k-blocks of weights a CTA pulls into L2 before its dependency wait.  Kept
// small: the SM's TMA unit works the prefetches off before the CTA's own loads,
// and deep prefetches delayed them (measured, step at B=1: 16 k-blocks 328 us,
// 4: 303 us, 2: 301 us, none: 306 us).
constexpr int kPrefetchKb = 2;
// K splits of one tile that reduce in a cluster: up to 16 (a non-portable
// cluster size, allowed per kernel).  Decode-sized projections have few weight
// tiles (fc, O and down of the GPT-OSS shape: 23) and need many splits each to
// give every SM several CTAs' worth of weight stream.
constexpr int kMaxClusterSplits = 16;
constexpr int kMaxPartialSplits = 16;       // splits storing their own partials
static_assert(kMaxPartialSplits <= 16, "the projection test hook holds 16 partial tiles");
// Weights are read in tile order (one contiguous 16 KB block per weight box;
// measured, LM head at B=1 with two CTAs per SM: 188 us packed, 192 us
// row-major).  Narrow token tiles stream weights: two 64-element K atoms per
// stage put the two 128-byte halves of each weight row's 256 bytes on the bus
// back to back (measured: LM head at B=1 259 us instead of 303 us).  Wide tiles
// keep one atom so that enough stages stay in flight.
constexpr int kNarrowBN = 64;
// Token tiles up to kOccBN wide run several CTAs per SM (see below), and no
// token tile is wider than kMaxBN.  Wide tiles gain from it too (measured, LM
// head at B=64, 448 tokens: 636 us with one CTA per SM, 535 us with two).  The
// token-tile width is the widest (up to kMaxBN) whose two ring stages fit a
// two-CTA share of an SM (measured: step at B=64 1207 -> 1168 us, the bf16-pair
// and dual GEMMs get two CTAs).
constexpr int kOccBN = 256;
constexpr int kMaxBN = 256;
// Narrow token tiles run several CTAs per SM, each with its share of the SM's
// shared memory: one CTA's loads keep only part of the SM's share of DRAM
// bandwidth busy, whatever its ring depth (measured, LM head of 201088 x 2880 at
// 8 tokens: 5 or 3 stages per CTA both 275 us; two CTAs of 3 stages 196 us,
// three of 3 one-atom stages 188 us).  Up to three per SM, fewer where two
// stages of a wide tile do not fit a third of the SM's shared memory.  (A 2-SM
// pair schedule, M = 256 MMAs over clusters of two CTAs, measured slower: LM
// head of 201088 x 2880 at 448 tokens 723 us as pairs, 459 us one-SM; one thread
// issuing tcgen05.mma keeps an SM's tensor pipe only about half busy whatever
// the instruction's M, so two issuing CTAs per SM beat one pair per two SMs.)
constexpr int kNarrowCtasPerSm = 3;
constexpr int kStreamCtasPerSm = 3;
// shared memory of an SM that its CTAs can have (228 KB less 1 KB)
constexpr size_t kSmemPerSm = 227 * 1024;
// per CTA beside its ring: the system's 1 KB, the static barriers and
// reduction buffers (under 1 KB), the ring's 1 KB alignment slack, and a
// margin; the vector-store instances also hold the epilogue warps' store
// scratch (8.25 KB)
constexpr size_t kCtaSmemOverhead = 5 * 1024;
constexpr size_t kEpiScratchBytes = 9 * 1024;
constexpr size_t cta_smem_overhead(bool vec) {
  return vec ? kCtaSmemOverhead + kEpiScratchBytes : kCtaSmemOverhead;
}
constexpr int kTcThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;

struct TcArgs {
  int M, K, N_cap, dual, bpair;
  int tile_base, tile_count;  // the (m, n) tiles of this launch
  int BN, n_tiles, m_tiles, k_splits, kb_per_split, num_kb, stages, acc_bufs;
  int atoms;  // 64-element K atoms per stage (a k-block is atoms * 64 elements)
  int k_atoms;  // 64-element atoms per weight row: box (m, atom) at row (m * k_atoms + atom) * 128
  uint32_t tmem_cols;
  const int* n_rows_dev;
  Epilogue epi;
  uint32_t* status;
};

// ------------------------------------------------------------------ epilogue math

template <typename T>
PE_DEV void epi_store_elem(const Epilogue& e, int f, int t, float v, float v2) {
  switch (e.mode) {
    case EPI_STORE:
      static_cast<T*>(e.out)[static_cast<size_t>(t) * e.ld_out + f] = Elem<T>::from_f(v);
      break;
    case EPI_STORE_F32:
    case EPI_PARTIAL_F32:  // (out already points at this split's partial tile)
      static_cast<float*>(e.out)[static_cast<size_t>(t) * e.ld_out + f] = v;
      break;
    case EPI_RESID_F32:
      static_cast<float*>(e.out)[static_cast<size_t>(t) * e.ld_out + f] =
          v + e.resid[static_cast<size_t>(t) * e.ld_resid + f];
      break;
    case EPI_SWIGLU: {
      const float s = v / (1.0f + expf(-v));
      static_cast<T*>(e.out)[static_cast<size_t>(t) * e.ld_out + f] = Elem<T>::from_f(s * v2);
      break;
    }
    case EPI_SWIGLU_PAIR: {
      const float h = v / (1.0f + expf(-v)) * v2;
      const bf16 hi = __float2bfloat16_rn(h);
      const size_t o = static_cast<size_t>(t) * e.ld_out + f;
      static_cast<bf16*>(e.out)[o] = hi;
      static_cast<bf16*>(e.out2)[o] = __float2bfloat16_rn(h - __bfloat162float(hi));
      break;
    }
    default:
      break;
  }
}

// Largest value over the warp (all lanes active); NaN if any lane holds NaN.
PE_DEV float warp_max_f32(float v) {
  float m;
  asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(m) : "f"(v));
  return m;
}

// Epilogue of 16 token columns j0..j0+15 for feature f (this thread's TMEM lane).
// ARGMAX: per column the warp takes the largest of its 32 features' values in
// one reduction and the first lane holding it from a ballot; lane i keeps
// column i's value and lane, builds its key, and the warp folds its 16 keys
// into the row maxima with one atomicMax each (no barrier across the epilogue
// warps).  Equal values resolve to the lowest feature, NaN counts as the
// largest (argmax_key orders the maxima of different warps the same way).
PE_DEV void tc_epilogue16(const TcArgs& p, const Epilogue& e, int f, int j0, const float* v,
                          const float* v2, int n_rows) {
  const bool fok = f < p.M;
  if (e.mode != EPI_ARGMAX) {
    if (!fok) return;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (j0 + i < n_rows) epi_store_elem<bf16>(e, f, j0 + i, v[i], v2 ? v2[i] : 0.f);
    return;
  }
  if (e.logits && fok) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (j0 + i < n_rows) e.logits[static_cast<size_t>(j0 + i) * e.ld_logits + f] = v[i];
  }
  const int lane = threadIdx.x & 31;
  float best = 0.f;
  uint32_t holders = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float x = fok ? v[i] : -INFINITY;
    const float m = warp_max_f32(x);
    const uint32_t hit = __ballot_sync(0xffffffffu, fok && (m != m ? x != x : x == m));
    if (lane == i) {
      best = m;
      holders = hit;
    }
  }
  if (lane < 16 && j0 + lane < n_rows && holders) {
    const int first = __ffs(static_cast<int>(holders)) - 1;
    atomicMax(&e.amax[j0 + lane], argmax_key(best, static_cast<uint32_t>(f - lane + first)));
  }
}

// Stores of a warp's 32 features x 16 token columns (j0..j0+15) with 4
// consecutive features per lane and instruction: the block passes through the
// warp's shared scratch w ([16][33] floats, padded rows: no bank conflicts), so
// each store instruction writes four token rows of 128 contiguous bytes rather
// than one.  (Measured, B=64 step: the partial-sum tiles of fc, QKV, O and down
// stored one float per lane: 1146 us; this way: 1091 us.)
constexpr int kEpiScratch = 16 * 33;  // floats per epilogue warp

// Whether the stores of epilogue `e` can go 4 features at a time: rows of a
// multiple of 4 elements and 16-byte aligned bases.
PE_DEV bool epi_vec_ok(const TcArgs& p, const Epilogue& e) {
  auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  if (e.mode == EPI_ARGMAX || (p.M & 3) || (e.ld_out & 3) || !al(e.out)) return false;
  if (e.mode == EPI_RESID_F32 && ((e.ld_resid & 3) || !al(e.resid))) return false;
  if (e.mode == EPI_SWIGLU_PAIR && !al(e.out2)) return false;
  return true;
}

// Four outputs of token row t, features fb..fb+3, from accumulator values x (and
// y, the second accumulator of the dual modes).
PE_DEV void epi_store4(const Epilogue& e, int t, int fb, const float* x, const float* y) {
  const size_t o = static_cast<size_t>(t) * e.ld_out + fb;
  switch (e.mode) {
    case EPI_STORE_F32:
    case EPI_PARTIAL_F32:  // (out already points at this split's partial tile)
      *reinterpret_cast<float4*>(static_cast<float*>(e.out) + o) =
          make_float4(x[0], x[1], x[2], x[3]);
      break;
    case EPI_RESID_F32: {
      const float4 r =
          *reinterpret_cast<const float4*>(e.resid + static_cast<size_t>(t) * e.ld_resid + fb);
      *reinterpret_cast<float4*>(static_cast<float*>(e.out) + o) =
          make_float4(x[0] + r.x, x[1] + r.y, x[2] + r.z, x[3] + r.w);
      break;
    }
    case EPI_STORE:
      *reinterpret_cast<uint2*>(static_cast<bf16*>(e.out) + o) =
          make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
      break;
    case EPI_SWIGLU: {
      float h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = x[k] / (1.0f + expf(-x[k])) * y[k];
      *reinterpret_cast<uint2*>(static_cast<bf16*>(e.out) + o) =
          make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
      break;
    }
    case EPI_SWIGLU_PAIR: {
      float h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = x[k] / (1.0f + expf(-x[k])) * y[k];
      uint32_t hi01, lo01, hi23, lo23;
      split_bf16x2(h[0], h[1], hi01, lo01);
      split_bf16x2(h[2], h[3], hi23, lo23);
      *reinterpret_cast<uint2*>(static_cast<bf16*>(e.out) + o) = make_uint2(hi01, hi23);
      *reinterpret_cast<uint2*>(static_cast<bf16*>(e.out2) + o) = make_uint2(lo01, lo23);
      break;
    }
    default:
      break;
  }
}

// f0: the warp's first feature; v (and v2 for dual modes): this lane's 16
// accumulator columns for feature f0 + lane.
PE_DEV void tc_store16_vec(const TcArgs& p, const Epilogue& e, int f0, int j0, const float* v,
                           const float* v2, int n_rows, float* w) {
  const int lane = threadIdx.x & 31;
  const int fq = (lane & 7) * 4;  // this lane's 4 features ...
  const int tr = lane >> 3;       // ... of token rows tr, tr + 4, tr + 8, tr + 12
  const int fb = f0 + fq;
  const bool live = fb < p.M;     // M is a multiple of 4: all four features or none
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i * 33 + lane] = v[i];
  __syncwarp();
  if (!v2) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      float x[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) x[k] = w[(tr + 4 * s) * 33 + fq + k];
      const int t = j0 + tr + 4 * s;
      if (live && t < n_rows) epi_store4(e, t, fb, x, nullptr);
    }
    __syncwarp();
    return;
  }
  float a[4][4];
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int k = 0; k < 4; ++k) a[s][k] = w[(tr + 4 * s) * 33 + fq + k];
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i * 33 + lane] = v2[i];
  __syncwarp();
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    float y[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = w[(tr + 4 * s) * 33 + fq + k];
    const int t = j0 + tr + 4 * s;
    if (live && t < n_rows) epi_store4(e, t, fb, a[s], y);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ tcgen05 kernel
//
// Two schedules share the kernel:
//  * k_splits == 1: persistent.  CTA b takes tiles b, b + grid, ... over
//    (m, n) tiles; two TMEM accumulators (when they fit) let the MMA of the
//    next tile run while the epilogue drains the current one.
//  * k_splits > 1: the splits of one (m, n) tile are one thread-block cluster
//    (rank = split).  Each CTA streams its share of K, parks its fp32 partial
//    tile in its own shared memory (the stage ring is idle by then), and after a
//    cluster barrier every CTA sums, over the cluster's ranks in rank order
//    (deterministic), the columns j with j % k_splits == rank, read through
//    distributed shared memory, and runs the epilogue on them.

struct TileRef {
  int m, n, ks;
};

// Tensor-map coordinates of the weight box of tile row m at reduction offset x
// (a multiple of 64).  Packed weights: past K the box lies beyond the last
// block, so TMA fills it with zeros as it does past K of a row-major weight.
PE_DEV void weight_box(const TcArgs& p, int m, int x, int& cx, int& cy) {
  const int a = x / kBK;
  cx = 0;
  cy = (a < p.k_atoms ? m * p.k_atoms + a : p.m_tiles * p.k_atoms) * kBM;
}

// The tile a CTA works on at its it-th turn; false when it has no more.
PE_DEV bool next_tile(const TcArgs& p, int it, TileRef& t) {
  if (p.k_splits > 1) {
    if (it > 0) return false;
    const int local = blockIdx.x / p.k_splits;
    if (local >= p.tile_count) return false;
    const int tile = p.tile_base + local;
    t.ks = blockIdx.x % p.k_splits;
    t.n = tile % p.n_tiles;
    t.m = tile / p.n_tiles;
    return t.m < p.m_tiles;
  }
  const int local = blockIdx.x + it * gridDim.x;
  if (local >= p.tile_count) return false;
  const int tile = p.tile_base + local;
  t.ks = 0;
  t.n = tile % p.n_tiles;
  t.m = tile / p.n_tiles;
  return true;
}

// A tile whose token rows all lie past the live row count is skipped, except a
// CTA's first tile when it is the token tile 0 (only an empty batch makes that
// one dead: every role then works through it the same way, and its epilogue
// stores nothing past the live rows).
PE_DEV bool tile_skipped(const TcArgs& p, const TileRef& t, int it, int n_rows) {
  return t.n * p.BN >= n_rows && !(it == 0 && t.n == 0);
}

// OCC: CTAs per SM the instance is launched for (each instance keeps its own
// fixed shared-memory limit, so graph replays of either stay launchable).
// VEC: the instance for token tiles of 32 rows or more at up to two CTAs per
// SM, whose stores go 4 features at a time through a shared scratch (the
// argmax epilogue and decode tiles of 16 rows keep the scalar instance:
// measured, LM head at B=64 458 us in it, 477 us in a shared one).
template <int OCC, bool VEC>
__global__ void __launch_bounds__(kTcThreads, OCC)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapA2,
                   const __grid_constant__ CUtensorMap mapB, const __grid_constant__ CUtensorMap mapB2,
                   const TcArgs p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], final_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, n_rows_sh;
  __shared__ unsigned long long red_sh[4];
  __shared__ int ep_ok[2][4];
  __shared__ float epi_sh[VEC ? 4 : 1][VEC ? kEpiScratch : 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int nA = p.dual ? 2 : 1;
  const int nB = p.bpair ? 2 : 1;
  const uint32_t b_bytes = static_cast<uint32_t>(p.BN) * 128u;
  const uint32_t atom_bytes = kABytes * nA + b_bytes * nB;
  const uint32_t stage_bytes = atom_bytes * p.atoms;
  const int kbk = kBK * p.atoms;  // elements of K per k-block
  const int nbuf = p.acc_bufs;
  const uint32_t buf_cols = static_cast<uint32_t>(p.BN * nA);
  // K splits reduce inside a cluster, unless each stores its own partial
  const bool clustered = p.k_splits > 1 && p.epi.mode != EPI_PARTIAL_F32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 128);
    }
    mbar_init(&final_bar, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mapA);
    if (p.dual) prefetch_tmap(&mapA2);
    prefetch_tmap(&mapB);
    if (p.bpair) prefetch_tmap(&mapB2);
    // The weights do not depend on the previous kernel: pull the first tile's
    // first k-blocks into L2 while that kernel finishes.  (Loading the first
    // stages' weight boxes straight into the ring before the dependency wait
    // measured 2-6 us slower per step at every workload.)
    TileRef t;
    if (next_tile(p, 0, t)) {
      const int kb0 = t.ks * p.kb_per_split;
      const int nkb = min(p.num_kb, kb0 + p.kb_per_split) - kb0;
      const int kb1 = min(kb0 + nkb, kb0 + kPrefetchKb / p.atoms);
      for (int kb = kb0; kb < kb1; ++kb)
        for (int at = 0; at < p.atoms; ++at) {
          if (kb * kbk + at * kBK >= p.K) break;
          int cx, cy;
          weight_box(p, t.m, kb * kbk + at * kBK, cx, cy);
          tma_prefetch_l2_2d(&mapA, cx, cy);
          if (p.dual) tma_prefetch_l2_2d(&mapA2, cx, cy);
        }
    }
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, p.tmem_cols);
    tmem_relinquish();
  }
  // the token rows, the row count and the epilogue's inputs come from earlier kernels
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) {
    int n = p.N_cap;
    if (p.n_rows_dev) {
      const int v = *p.n_rows_dev;
      n = v < 0 ? 0 : (v < n ? v : n);
    }
    n_rows_sh = n;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = tmem_base_sh;
  const int n_rows = n_rows_sh;
  volatile int* abort_flag = &abort_sh;
  auto fail = [&]() {
    abort_sh = 1;
    set_status(p.status, PE_ST_TIMEOUT);
  };
  // cluster mode: this CTA's partial tile, [acc][column][128 features] fp32,
  // parked at the start of the (by then idle) stage ring
  float* part = reinterpret_cast<float*>(smem);

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      // per stage: ever armed / parity of the last arm
      uint32_t armed = 0u, armed_parity = 0;
      auto issue_b = [&](int s, int kb, int tn) {
        for (int at = 0; at < p.atoms; ++at) {
          uint8_t* sa = smem + static_cast<size_t>(s) * stage_bytes + at * atom_bytes;
          const int x = kb * kbk + at * kBK;
          tma_load_2d(sa + kABytes * nA, &mapB, &full_bar[s], x, tn * p.BN, pol_x);
          if (p.bpair)
            tma_load_2d(sa + kABytes * nA + b_bytes, &mapB2, &full_bar[s], x, tn * p.BN, pol_x);
        }
      };
      TileRef t;
      for (int it = 0; next_tile(p, it, t) && !*abort_flag; ++it) {
        if (tile_skipped(p, t, it, n_rows)) continue;
        const int kb0 = t.ks * p.kb_per_split;
        const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag)) {
            fail();
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], stage_bytes);
          // the atoms of one row follow each other in memory: their boxes go
          // out back to back, A first (the weights dominate the traffic)
          for (int at = 0; at < p.atoms; ++at) {
            uint8_t* sa = smem + static_cast<size_t>(stage) * stage_bytes + at * atom_bytes;
            int cx, cy;
            weight_box(p, t.m, kb * kbk + at * kBK, cx, cy);
            tma_load_2d(sa, &mapA, &full_bar[stage], cx, cy, pol_w);
            if (p.dual) tma_load_2d(sa + kABytes, &mapA2, &full_bar[stage], cx, cy, pol_w);
          }
          issue_b(stage, kb, t.n);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory goes away
        for (int s = 0; s < p.stages; ++s)
          if (armed & (1u << s)) {
            int dummy = 0;
            mbar_wait(&full_bar[s], (armed_parity >> s) & 1u, &dummy);
          }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, p.BN);
      int stage = 0, cnt = 0;
      uint32_t phase = 0, acc_phase[2] = {0u, 0u};
      TileRef t;
      for (int it = 0; next_tile(p, it, t) && !*abort_flag; ++it) {
        if (tile_skipped(p, t, it, n_rows)) continue;
        const int b = cnt % nbuf;
        ++cnt;
        const int kb0 = t.ks * p.kb_per_split;
        const int kb1 = min(p.num_kb, kb0 + p.kb_per_split);
        if (!mbar_wait(&tempty_bar[b], acc_phase[b] ^ 1u, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(b) * buf_cols;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          for (int at = 0; at < p.atoms; ++at) {
          const uint32_t sa =
              smem_u32(smem + static_cast<size_t>(stage) * stage_bytes + at * atom_bytes);
          const uint64_t adesc = sw128_kmajor_desc(sa);
          const uint64_t a2desc = sw128_kmajor_desc(sa + kABytes);
          const uint64_t bdesc = sw128_kmajor_desc(sa + kABytes * nA);
          const uint64_t b2desc = sw128_kmajor_desc(sa + kABytes * nA + b_bytes);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // advance 16 elements (32 bytes) along K inside the swizzle row
            const uint32_t acc = (kb > kb0 || at > 0 || kk > 0) ? 1u : 0u;
            umma_bf16(d0, adesc + 2 * kk, bdesc + 2 * kk, idesc, acc);
            if (p.bpair) umma_bf16(d0, adesc + 2 * kk, b2desc + 2 * kk, idesc, 1u);
            if (p.dual) {
              const uint32_t d1 = d0 + static_cast<uint32_t>(p.BN);
              umma_bf16(d1, a2desc + 2 * kk, bdesc + 2 * kk, idesc, acc);
              if (p.bpair) umma_bf16(d1, a2desc + 2 * kk, b2desc + 2 * kk, idesc, 1u);
            }
          }
          }
          umma_commit(&empty_bar[stage]);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[b]);
        acc_phase[b] ^= 1u;
      }
      // every MMA issued by this thread has finished before TMEM is released
      umma_commit(&final_bar);
      int dummy = 0;
      mbar_wait(&final_bar, 0, &dummy);
    }
  } else {
    // ---------------- epilogue warps 2..5: TMEM lane quarter = warp % 4
    const int q = warp & 3;
    const int ew = warp - 2;
    const int fl = q * 32 + lane;  // this thread's feature within the tile
    uint32_t acc_phase[2] = {0u, 0u};
    int cnt = 0;
    TileRef t;
    for (int it = 0; next_tile(p, it, t) && !*abort_flag; ++it) {
      if (tile_skipped(p, t, it, n_rows)) continue;
      const int b = cnt % nbuf;
      const int par = cnt & 1;
      ++cnt;
      // the four epilogue warps decide together whether to go on, so none of
      // them can be left waiting at a named barrier the others skipped
      const bool ok = mbar_wait(&tfull_bar[b], acc_phase[b], abort_flag);
      if (lane == 0) ep_ok[par][ew] = ok ? 1 : 0;
      named_bar_sync(1, 128);
      if (!(ep_ok[par][0] && ep_ok[par][1] && ep_ok[par][2] && ep_ok[par][3])) {
        fail();
        break;
      }
      acc_phase[b] ^= 1u;
      tc_fence_after();
      const int f = t.m * kBM + fl;
      const int jt = t.n * p.BN;
      const uint32_t tl = tmem_base + static_cast<uint32_t>(b) * buf_cols +
                          (static_cast<uint32_t>(q * 32) << 16);
      if (!clustered) {
        Epilogue ep = p.epi;
        if (ep.mode == EPI_PARTIAL_F32)
          ep.out = static_cast<float*>(ep.out) + static_cast<size_t>(t.ks) * ep.part_stride;
        const bool vec = VEC && epi_vec_ok(p, ep);
        for (int c = 0; c < p.BN; c += 16) {
          float v[16], v2[16];
          tmem_ld16(tl + c, v);
          if (p.dual) tmem_ld16(tl + p.BN + c, v2);
          if (c + 16 >= p.BN) {
            // last TMEM read of this buffer: hand it back before the stores
            tc_fence_before();
            mbar_arrive(&tempty_bar[b]);
          }
          if constexpr (VEC) {
            if (vec) {
              tc_store16_vec(p, ep, f - lane, jt + c, v, p.dual ? v2 : nullptr, n_rows,
                             epi_sh[ew]);
              continue;
            }
          }
          tc_epilogue16(p, ep, f, jt + c, v, p.dual ? v2 : nullptr, n_rows);
        }
      } else {
        // park the partial tile: part[a][j][fl] (consecutive features, conflict-free)
        for (int c = 0; c < p.BN; c += 16) {
          float v[16];
          tmem_ld16(tl + c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) part[(c + i) * kBM + fl] = v[i];
          if (p.dual) {
            tmem_ld16(tl + p.BN + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) part[(p.BN + c + i) * kBM + fl] = v[i];
          }
        }
        tc_fence_before();
      }
    }
  }

  if (clustered) {
    // every CTA of the cluster has parked its partial (a CTA that gave up on a
    // wait leaves its partial unwritten; its status bit reports the problem) ...
    __syncwarp();
    cluster_sync_all();
    if (warp >= 2 && !*abort_flag) {
      const int fl = (warp & 3) * 32 + lane;
      TileRef t;
      if (next_tile(p, 0, t) && !tile_skipped(p, t, 0, n_rows)) {
        const int f = t.m * kBM + fl;
        const int jt = t.n * p.BN;
        const uint32_t rank = cluster_ctarank();
        const uint32_t base = smem_u32(part);
        const int ew = warp - 2, et = threadIdx.x - 64;
        for (int j = static_cast<int>(rank); j < p.BN; j += p.k_splits) {
          if (jt + j >= n_rows) break;  // uniform over the epilogue warps
          // all the splits' loads go out before the first add (they are
          // independent); the sum still runs in rank order
          float pv[kMaxClusterSplits], pv2[kMaxClusterSplits];
          const uint32_t o1 = base + static_cast<uint32_t>((j * kBM + fl) * 4);
          const uint32_t o2 = base + static_cast<uint32_t>(((p.BN + j) * kBM + fl) * 4);
#pragma unroll
          for (int r = 0; r < kMaxClusterSplits; ++r) {
            if (r < p.k_splits) {
              pv[r] = ld_dsmem_f32(o1, r);
              pv2[r] = p.dual ? ld_dsmem_f32(o2, r) : 0.f;
            }
          }
          float v = 0.f, v2 = 0.f;
#pragma unroll
          for (int r = 0; r < kMaxClusterSplits; ++r) {
            if (r < p.k_splits) {
              v += pv[r];
              v2 += pv2[r];
            }
          }
          if (p.epi.mode == EPI_ARGMAX) {
            // max over this tile's 128 features of token jt + j
            if (p.epi.logits && f < p.M)
              p.epi.logits[static_cast<size_t>(jt + j) * p.epi.ld_logits + f] = v;
            const unsigned long long k = warp_max_u64(f < p.M ? argmax_key(v, f) : 0ull);
            if (lane == 0) red_sh[ew] = k;
            named_bar_sync(1, 128);
            if (et == 0) {
              unsigned long long kk = red_sh[0];
              for (int w2 = 1; w2 < 4; ++w2) kk = red_sh[w2] > kk ? red_sh[w2] : kk;
              if (kk) atomicMax(&p.epi.amax[jt + j], kk);
            }
            named_bar_sync(1, 128);
          } else if (f < p.M) {
            epi_store_elem<bf16>(p.epi, f, jt + j, v, v2);
          }
        }
      }
    }
    // ... and no CTA leaves while another may still read its shared memory
    __syncwarp();
    cluster_sync_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// ------------------------------------------------------------------ host: plan + launch

static_assert(kNarrowCtasPerSm >= 1 && kNarrowCtasPerSm <= 3, "CTAs per SM");
static_assert(kStreamCtasPerSm >= 1 && kStreamCtasPerSm <= 3, "CTAs per SM");
using TcKernelFn = decltype(&gemm_tc_kernel<1, false>);

// The instance for `occ` CTAs per SM, with vector stores or not (these exist
// for up to two CTAs per SM).
static TcKernelFn tc_kernel(int occ, bool vec) {
  if (vec && occ <= 2) return occ == 2 ? gemm_tc_kernel<2, true> : gemm_tc_kernel<1, true>;
  return occ >= 3 ? gemm_tc_kernel<3, false>
                  : occ == 2 ? gemm_tc_kernel<2, false> : gemm_tc_kernel<1, false>;
}

// Dynamic shared memory limit of an instance: its largest ring plus the 1 KB
// alignment slack.  The limit, not a launch's own size, decides how many CTAs
// of the function the SM takes, so it is what makes `occ` CTAs fit.
static size_t tc_max_dyn_smem(int occ, bool vec) {
  return occ > 1 ? kSmemPerSm / occ - cta_smem_overhead(vec) + 1024 : kSmemBudget + 1024;
}

// Set the attributes of the `occ` instances: the same values at every launch.
static cudaError_t tc_prepare(int occ) {
  cudaError_t e = cudaSuccess;
  for (const bool vec : {false, true}) {
    if (vec && occ > 2) continue;
    const TcKernelFn k = tc_kernel(occ, vec);
    cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(tc_max_dyn_smem(occ, vec)));
    if (r != cudaSuccess) e = r;
    r = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (r != cudaSuccess) e = r;
    cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
  }
  return e;
}

// How many clusters of `cs` CTAs of the `occ` instance with `smem` bytes each
// can be resident at once.  The query places one CTA of this kernel per SM (as
// the per-SM query does); `occ` such placements side by side fit as well, so
// its answer times `occ` is a lower bound on what the SMs hold.
static int max_active_clusters(int occ, int cs, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<std::pair<int, int>, size_t>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(std::make_pair(occ, cs), smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  tc_prepare(occ);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs * 64);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (void*)tc_kernel(occ, false), &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[key] = n * occ;
  return n * occ;
}

TcPlan plan_gemm_tc(int M, int K, int N_cap, int dual, int bpair, int num_sms, bool allow_split,
                    bool partial) {
  TcPlan pl{};
  pl.M = M;
  pl.K = K;
  pl.N_cap = N_cap < 1 ? 1 : N_cap;
  pl.dual = dual;
  pl.bpair = bpair;
  const int nA = dual ? 2 : 1;
  const int nB = bpair ? 2 : 1;
  // token tile: at most kMaxBN rows, and narrow enough that three stages fit
  int nt = (pl.N_cap + kMaxBN - 1) / kMaxBN;
  size_t stage_bytes = 0;
  for (;; ++nt) {
    int bn = (pl.N_cap + nt - 1) / nt;
    bn = (bn + 15) / 16 * 16;
    pl.BN = bn < 16 ? 16 : bn;
    pl.atoms = pl.BN <= kNarrowBN ? 2 : 1;
    stage_bytes = (static_cast<size_t>(kABytes) * nA + static_cast<size_t>(pl.BN) * 128 * nB) *
                  pl.atoms;
    // wide enough, but two stages fit a two-CTA share of the SM
    if ((kSmemPerSm / 2 - cta_smem_overhead(true)) / stage_bytes >= 2 || pl.BN <= 64) break;
  }
  pl.n_tiles = (pl.N_cap + pl.BN - 1) / pl.BN;
  pl.m_tiles = (M + kBM - 1) / kBM;
  // CTAs per SM: narrow tiles share each SM among several CTAs of at least two
  // stages each (fewer atoms per stage where that is what fits); a stream of at
  // least two full rounds of tiles takes the most
  // token tiles of 32 rows or more take the vector-store instances (their
  // scratch comes out of the ring's share) where they run at most two CTAs per
  // SM; decode tiles of 16 rows keep the ring (measured, B=1 step: 3 us more
  // with one stage less for gate/up)
  const bool wide = pl.BN >= 32;
  int occ = 1;
  size_t budget = kSmemBudget;
  if (pl.BN <= kOccBN) {
    const int want = pl.m_tiles * pl.n_tiles >= 2 * kStreamCtasPerSm * num_sms ? kStreamCtasPerSm
                                                                                : kNarrowCtasPerSm;
    // the most CTAs per SM (down from `want`) that still get two stages each
    for (int o = want; o >= 2 && occ == 1; --o) {
      const size_t b = tc_max_dyn_smem(o, wide && o <= 2) - 1024;
      int atoms = pl.atoms;
      size_t sb = stage_bytes;
      while (atoms > 1 && b / sb < 2) {
        atoms /= 2;
        sb = (static_cast<size_t>(kABytes) * nA + static_cast<size_t>(pl.BN) * 128 * nB) * atoms;
      }
      if (b / sb >= 2) {
        occ = o;
        budget = b;
        pl.atoms = atoms;
        stage_bytes = sb;
      }
    }
  }
  pl.num_kb = (K + kBK * pl.atoms - 1) / (kBK * pl.atoms);
  const int stages = static_cast<int>(budget / stage_bytes);
  pl.stages = std::max(2, std::min(kMaxStages, stages));
  pl.smem_bytes = pl.stages * stage_bytes + 1024;
  // (the occupancy query answers 1 for this kernel at any size, though the SM
  // does run two such CTAs side by side: the fit is the arithmetic above, and
  // no CTA outside a cluster waits for another, so it is only a speed matter)
  pl.ctas_per_sm = occ;
  pl.vec = wide && occ <= 2 ? 1 : 0;
  // the resident CTAs of one wave; every "SM" count below is in these slots
  num_sms *= occ;
  const int base = pl.m_tiles * pl.n_tiles;
  // split K across a cluster when one wave of plain tiles leaves SMs idle: the
  // splits of a tile must all be resident at once, their partial tile must fit
  // in the stage ring, and at least 4 k-blocks go to each split
  // Partial sums pay for wide token tiles (their consumer adds a few splits);
  // narrow decode tiles split many ways and reduce in a cluster instead
  // (measured, step at B=1: 297 us with the cluster reduction, 305 us with 13
  // partial tiles per projection; at B=64 the partial sums save 20 us).
  partial = partial && pl.BN > kNarrowBN;
  pl.partial = partial ? 1 : 0;
  int s = 1;
  if (allow_split && base < num_sms && partial) {
    // each split stores its own partial sum: as many as fill the CTA slots
    s = std::min(kMaxPartialSplits, num_sms / base);
    s = std::min(s, pl.num_kb * pl.atoms / 4);
    if (s < 2) s = 1;
  } else if (allow_split && base < num_sms) {
    s = std::min(kMaxClusterSplits, num_sms / base);
    s = std::min(s, pl.num_kb * pl.atoms / 4);
    const size_t part_bytes = static_cast<size_t>(nA) * pl.BN * kBM * sizeof(float);
    if (part_bytes > pl.stages * stage_bytes) s = 1;
    while (s > 1 && max_active_clusters(occ, s, pl.smem_bytes) * s < base * s) --s;
    if (s < 2) s = 1;
  }
  pl.kb_per_split = (pl.num_kb + s - 1) / s;
  pl.k_splits = (pl.num_kb + pl.kb_per_split - 1) / pl.kb_per_split;
  pl.acc_bufs = (pl.k_splits == 1 && 2 * pl.BN * nA <= 512) ? 2 : 1;
  // TMEM columns: a power of two >= 32; the CTAs sharing an SM share its 512
  auto tmem_cols_for = [&](int bufs) {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(bufs * pl.BN * nA)) c <<= 1;
    return static_cast<int>(c);
  };
  if (tmem_cols_for(pl.acc_bufs) * occ > 512) pl.acc_bufs = 1;
  pl.tmem_cols = tmem_cols_for(pl.acc_bufs);
  pl.grid = pl.k_splits > 1 ? base * pl.k_splits : std::min(base, num_sms);
  pl.main_tiles = base;
  pl.tail_splits = 1;
  pl.tail_kb_per_split = pl.num_kb;
  if (pl.k_splits == 1 && base > num_sms && !partial) {
    // Several rounds of persistent tiles: a partial last round leaves SMs idle
    // while a few CTAs finish one more tile.  Run the full rounds persistent and
    // the remaining tiles as clusters that split them over K.
    const int rem = base % num_sms;
    int ts = rem ? std::min(kMaxClusterSplits, num_sms / rem) : 1;
    ts = std::min(ts, pl.num_kb * pl.atoms / 4);
    const size_t part_bytes = static_cast<size_t>(nA) * pl.BN * kBM * sizeof(float);
    if (part_bytes > pl.stages * stage_bytes) ts = 1;
    while (ts > 1 && max_active_clusters(occ, ts, pl.smem_bytes) < rem) --ts;
    if (ts >= 2) {
      pl.main_tiles = base - rem;
      pl.tail_kb_per_split = (pl.num_kb + ts - 1) / ts;
      pl.tail_splits = (pl.num_kb + pl.tail_kb_per_split - 1) / pl.tail_kb_per_split;
    }
  }
  return pl;
}

// One launch over tiles [tile_base, tile_base + tile_count) with k_splits splits
// of kb_per_split k-blocks each (k_splits > 1: clusters of k_splits CTAs).
static int launch_one(const TcPlan& pl, const CUtensorMap* mapA, const CUtensorMap* mapA2,
                      const CUtensorMap& mapB, const CUtensorMap& mapB2, const int* n_rows_dev,
                      const Epilogue& epi, uint32_t* status, cudaStream_t st, int tile_base,
                      int tile_count, int k_splits, int kb_per_split, int grid) {
  TcArgs a{};
  a.M = pl.M;
  a.K = pl.K;
  a.N_cap = pl.N_cap;
  a.dual = pl.dual;
  a.bpair = pl.bpair;
  a.tile_base = tile_base;
  a.tile_count = tile_count;
  a.BN = pl.BN;
  a.n_tiles = pl.n_tiles;
  a.m_tiles = pl.m_tiles;
  a.k_splits = k_splits;
  a.k_atoms = (pl.K + kBK - 1) / kBK;
  a.kb_per_split = kb_per_split;
  a.num_kb = pl.num_kb;
  a.atoms = pl.atoms;
  a.stages = pl.stages;
  a.acc_bufs = k_splits == 1 ? pl.acc_bufs : 1;
  a.tmem_cols = static_cast<uint32_t>(pl.tmem_cols);
  a.n_rows_dev = n_rows_dev;
  a.epi = epi;
  a.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = pl.smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = k_splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (k_splits > 1 && epi.mode != EPI_PARTIAL_F32) ? 2 : 1;
  // the vector-store instance for the stores of a wide tile; the argmax
  // epilogue and cluster-reduced splits take the scalar one
  const bool vec = pl.vec && epi.mode != EPI_ARGMAX && cfg.numAttrs == 1;
  return cudaLaunchKernelEx(&cfg, tc_kernel(pl.ctas_per_sm, vec), *mapA,
                            pl.dual ? *mapA2 : *mapA, mapB,
                            mapB2, a) ==
                 cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}

int launch_gemm_tc(const TcPlan& pl, const CUtensorMap* mapA, const CUtensorMap* mapA2,
                   const void* X, const void* X_lo, const int* n_rows_dev, const Epilogue& epi,
                   uint32_t* status, cudaStream_t st) {
  if (pl.dual && !mapA2) return PE_ERR_ARG;
  if (pl.bpair && !X_lo) return PE_ERR_ARG;
  const uint32_t b_box = static_cast<uint32_t>(pl.BN);
  CUtensorMap mapB, mapB2;
  if (!encode_tmap_bf16(&mapB, X, static_cast<uint64_t>(pl.N_cap), static_cast<uint64_t>(pl.K),
                        b_box))
    return PE_ERR_CUDA;
  if (pl.bpair) {
    if (!encode_tmap_bf16(&mapB2, X_lo, static_cast<uint64_t>(pl.N_cap),
                          static_cast<uint64_t>(pl.K), b_box))
      return PE_ERR_CUDA;
  } else {
    mapB2 = mapB;
  }
  // one attribute value per instance for every launch, so kernels captured
  // into a graph stay launchable whatever order they replay in
  if (tc_prepare(pl.ctas_per_sm) != cudaSuccess) return PE_ERR_CUDA;
  const int base = pl.m_tiles * pl.n_tiles;
  if (pl.k_splits > 1)
    return launch_one(pl, mapA, mapA2, mapB, mapB2, n_rows_dev, epi, status, st, 0, base,
                      pl.k_splits, pl.kb_per_split, pl.grid);
  int rc = launch_one(pl, mapA, mapA2, mapB, mapB2, n_rows_dev, epi, status, st, 0, pl.main_tiles,
                      1, pl.num_kb, std::min(pl.main_tiles, pl.grid));
  if (rc != PE_OK || pl.main_tiles == base) return rc;
  const int tail = base - pl.main_tiles;
  return launch_one(pl, mapA, mapA2, mapB, mapB2, n_rows_dev, epi, status, st, pl.main_tiles, tail,
                    pl.tail_splits, pl.tail_kb_per_split, tail * pl.tail_splits);
}

// ------------------------------------------------------------------ fp32 SIMT kernel

constexpr int kSt = 64;  // tile edge (features x tokens)
constexpr int kSk = 16;  // reduction chunk

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ W,
                                                       const float* __restrict__ W2,
                                                       const float* __restrict__ X, int M, int K,
                                                       int N_cap, const int* n_rows_dev,
                                                       Epilogue e) {
  __shared__ float Ws[kSk][kSt + 1];
  __shared__ float W2s[kSk][kSt + 1];
  __shared__ float Xs[kSk][kSt + 1];
  pdl_trigger();
  pdl_wait();
  int n_rows = N_cap;
  if (n_rows_dev) n_rows = min(max(*n_rows_dev, 0), N_cap);
  const int f0 = blockIdx.x * kSt, t0 = blockIdx.y * kSt;
  if (t0 >= n_rows) return;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool dual = W2 != nullptr;
  float acc[4][4] = {}, acc2[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kSk) {
    for (int i = threadIdx.x; i < kSt * kSk; i += 256) {
      const int r = i / kSk, kk = i % kSk;
      const int f = f0 + r, t = t0 + r, k = k0 + kk;
      Ws[kk][r] = (f < M && k < K) ? W[static_cast<size_t>(f) * K + k] : 0.f;
      if (dual) W2s[kk][r] = (f < M && k < K) ? W2[static_cast<size_t>(f) * K + k] : 0.f;
      Xs[kk][r] = (t < n_rows && k < K) ? X[static_cast<size_t>(t) * K + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSk; ++kk) {
      float wv[4], w2v[4], xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wv[i] = Ws[kk][tx * 4 + i];
        w2v[i] = dual ? W2s[kk][tx * 4 + i] : 0.f;
        xv[i] = Xs[kk][ty * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(wv[i], xv[j], acc[i][j]);
          acc2[i][j] = fmaf(w2v[i], xv[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int t = t0 + ty * 4 + j;
    if (t >= n_rows) continue;
    if (e.mode == EPI_ARGMAX) {
      unsigned long long best = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int f = f0 + tx * 4 + i;
        if (f >= M) continue;
        if (e.logits) e.logits[static_cast<size_t>(t) * e.ld_logits + f] = acc[i][j];
        const unsigned long long k = argmax_key(acc[i][j], f);
        best = k > best ? k : best;
      }
      if (best) atomicMax(&e.amax[t], best);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int f = f0 + tx * 4 + i;
        if (f < M) epi_store_elem<float>(e, f, t, acc[i][j], acc2[i][j]);
      }
    }
  }
}

int launch_gemm_f32(const float* W, const float* W2, const float* X, int M, int K, int N_cap,
                    const int* n_rows_dev, const Epilogue& epi, cudaStream_t st) {
  if (N_cap <= 0 || M <= 0) return PE_OK;
  dim3 grid((M + kSt - 1) / kSt, (N_cap + kSt - 1) / kSt);
  return launch_pdl(gemm_f32_kernel, grid, dim3(256), 0, st, W, W2, X, M, K, N_cap, n_rows_dev,
                    epi) == cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}

// ------------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool encode_tmap_bf16(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !ptr || rows == 0 || cols == 0 || (cols % 8) != 0) return false;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ tile-packed weights

size_t packed_weight_bytes(int M, int K) {
  const size_t mt = static_cast<size_t>((M + kBM - 1) / kBM);
  const size_t ka = static_cast<size_t>((K + kBK - 1) / kBK);
  return mt * ka * kABytes;
}

// One thread per 16-byte chunk of the packed copy: chunk c of row r of block
// (m, a) holds W[128m + r][64a + 8c .. 64a + 8c + 7] (zeros past M or K; K is a
// multiple of 8, so a chunk is all in or all out).
__global__ void pack_weight_kernel(const uint4* __restrict__ W, int M, int K, int k_atoms,
                                   size_t n_chunks, uint4* __restrict__ P) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_chunks;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i & 7);
    const size_t rowi = i >> 3;  // row of the packed [blocks * 128][64] view
    const int r = static_cast<int>(rowi % kBM);
    const size_t blk = rowi / kBM;
    const int a = static_cast<int>(blk % k_atoms);
    const int m = static_cast<int>(blk / k_atoms);
    const int f = m * kBM + r;
    const int k = a * kBK + c * 8;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (f < M && k < K) v = W[(static_cast<size_t>(f) * K + k) / 8];
    P[i] = v;
  }
}

int pack_weight(const void* W, int M, int K, void* P, cudaStream_t st) {
  if (!W || !P || M <= 0 || K <= 0 || K % 8) return PE_ERR_ARG;
  const size_t n_chunks = packed_weight_bytes(M, K) / 16;
  const int k_atoms = (K + kBK - 1) / kBK;
  const size_t blocks = std::min<size_t>((n_chunks + 255) / 256, 152u * 16u);
  pack_weight_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(
      static_cast<const uint4*>(W), M, K, k_atoms, n_chunks, static_cast<uint4*>(P));
  return cudaGetLastError() == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

bool encode_packed_weight_map(CUtensorMap* map, const void* P, int M, int K) {
  const uint64_t rows = packed_weight_bytes(M, K) / 128;
  return encode_tmap_bf16(map, P, rows, 64, static_cast<uint32_t>(kBM));
}


int num_sms_of_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace pe
