// Paged attention of the K draft queries of each request over its whole
// context plus the earlier draft positions ("P-EAGLE: parallel speculative
// decoding in vLLM", Parallel drafting: all positions pass through the layer at
// once; draft position k sees every cache position up to its own).
//
// bf16: one CTA per (request, KV head, key split).  Its query tile is the K
// sample rows x the H/G query heads that share the KV head (GQA), 16 rows per
// warp.  Keys stream through shared memory in chunks of 64 (cp.async, 3 stages,
// 16-byte chunks XOR-swizzled by row so ldmatrix is conflict-free); S = Q K^T and
// O += P V run on warp-level bf16 mma.sync with fp32 accumulators and an online
// softmax in the exp2 domain (P enters the second product as a hi + lo bf16 pair).  Each split writes unnormalised partials; a combine
// kernel merges the splits (flash-decoding style).
//
// fp32: one CTA per (sample row, query head), SIMT dot products, online softmax.
#include <algorithm>
#include <cmath>

#include "pe_common.cuh"
#include "pe_prep.h"

namespace pe {

constexpr int kKC = 64;  // keys per chunk
// cp.async ring depth: three chunks for hd 64; two for hd 128, whose 32 KB
// chunks would otherwise hold an SM to two CTAs
template <int HD>
__host__ __device__ constexpr int ring_stages() {
  return HD >= 128 ? 2 : 3;
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 128;       // key splits per (request, KV head)
constexpr long kMaxSplitKeys = 2048;  // keys per split, at most

template <int HD>
__global__ void __launch_bounds__(256) attn_mma_kernel(const AttnArgs a) {
  constexpr int kStages = ring_stages<HD>();
  constexpr int ROWB = HD * 2;       // bytes per key row in shared memory
  constexpr int CH = HD / 8;         // 16-byte chunks per key row
  constexpr int TILE = kKC * ROWB;   // one K or V chunk
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_trigger();
  pdl_wait();
  const int split = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
  const int HG = a.H / a.G;
  const int rows = a.K * HG;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;

  int L = a.seq_len[r];
  const int Lmax = a.max_blocks * a.bs;
  if (L > Lmax || L < a.K) {
    if (threadIdx.x == 0) set_status(a.status, PE_ST_BLOCK_RANGE);
    L = min(max(L, 0), Lmax);
  }
  const int P0 = L - a.K;  // position of the first draft query (the NTP row)
  const int t0 = split * a.split_len;
  const int t1 = min(L, t0 + a.split_len);
  const size_t n_samp = static_cast<size_t>(a.B) * a.K;

  // rows handled by this thread: ra = 16*warp + gq, rb = ra + 8
  const int ra = warp * 16 + gq, rb = ra + 8;
  auto row_sample = [&](int row) { return static_cast<size_t>(r) * a.K + row / HG; };
  auto row_head = [&](int row) { return g * HG + row % HG; };

  if (t0 >= t1) {
    for (int hf = 0; hf < 2; ++hf) {
      const int rr = hf ? rb : ra;
      if (rr >= rows) continue;
      const size_t idx = (static_cast<size_t>(split) * n_samp + row_sample(rr)) * a.H + row_head(rr);
      if (tq == 0) {
        a.part_ml[idx * 2] = -INFINITY;
        a.part_ml[idx * 2 + 1] = 0.f;
      }
      for (int d = tq * 2; d < HD; d += 8) {
        a.part_o[idx * HD + d] = 0.f;
        a.part_o[idx * HD + d + 1] = 0.f;
      }
    }
    return;
  }

  // Q fragments (A operand of m16n8k16, row-major), zero for padding rows
  uint32_t qf[HD / 16][4];
  {
    const bf16* q = static_cast<const bf16*>(a.q);
    auto qrow = [&](int row) -> const bf16* {
      return row < rows ? q + (row_sample(row) * a.H + row_head(row)) * HD : nullptr;
    };
    const bf16* qa = qrow(ra);
    const bf16* qb = qrow(rb);
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

  const bf16* kc = static_cast<const bf16*>(a.k_cache);
  const bf16* vc = static_cast<const bf16*>(a.v_cache);
  const uint32_t sbase = smem_u32(smem);
  const int n_chunks = (t1 - t0 + kKC - 1) / kKC;

  auto load_chunk = [&](int c, int stage) {
    const uint32_t kdst = sbase + stage * 2 * TILE;
    const uint32_t vdst = kdst + TILE;
    for (int idx = threadIdx.x; idx < kKC * CH; idx += blockDim.x) {
      const int key = idx / CH, ch = idx - key * CH;
      const int t = t0 + c * kKC + key;
      bool ok = t < t1;
      size_t off = 0;
      if (ok) {
        const int blk = a.block_table[static_cast<size_t>(r) * a.max_blocks + t / a.bs];
        if (blk < 0 || blk >= a.num_blocks) {
          set_status(a.status, PE_ST_BLOCK_RANGE);
          ok = false;
        } else {
          off = ((static_cast<size_t>(blk) * a.G + g) * a.bs + t % a.bs) * HD + ch * 8;
        }
      }
      const uint32_t so = key * ROWB + ((ch ^ (key & 7)) << 4);
      cp_async16(kdst + so, kc + off, ok);
      cp_async16(vdst + so, vc + off, ok);
    }
  };

  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  const float sc = kLog2e / sqrtf(static_cast<float>(HD));

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < n_chunks) load_chunk(s, s);
    cp_async_commit();
  }

  for (int c = 0; c < n_chunks; ++c) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int nc = c + kStages - 1;
      if (nc < n_chunks) load_chunk(nc, nc % kStages);
      cp_async_commit();
    }
    const uint32_t ks_base = sbase + (c % kStages) * 2 * TILE;
    const uint32_t vs_base = ks_base + TILE;

    // S = Q K^T over 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
      for (int nt = 0; nt < 8; nt += 2) {
        const int mat = lane >> 3;
        const int key = nt * 8 + (mat >> 1) * 8 + (lane & 7);
        const int ch = ks * 2 + (mat & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(ks_base + key * ROWB + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_16816(s[nt], qf[ks], b0, b1);
        mma_bf16_16816(s[nt + 1], qf[ks], b2, b3);
      }
    }
    // scale, causal / range mask, online softmax (rows ra: s[.][0..1], rb: s[.][2..3])
    const int kbase = t0 + c * kKC;
    float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = kbase + nt * 8 + tq * 2 + e;
        const bool valid = t < t1;
        s[nt][e] = (valid && t <= lim_a) ? s[nt][e] * sc : -INFINITY;
        s[nt][2 + e] = (valid && t <= lim_b) ? s[nt][2 + e] * sc : -INFINITY;
        mx_a = fmaxf(mx_a, s[nt][e]);
        mx_b = fmaxf(mx_b, s[nt][2 + e]);
      }
    }
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
    mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
    mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float al_a = (mn_a == -INFINITY) ? 1.f : exp2f(m_a - mn_a);
    const float al_b = (mn_b == -INFINITY) ? 1.f : exp2f(m_b - mn_b);
    m_a = mn_a;
    m_b = mn_b;
    float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s[nt][e] = (mn_a == -INFINITY) ? 0.f : exp2f(s[nt][e] - mn_a);
        s[nt][2 + e] = (mn_b == -INFINITY) ? 0.f : exp2f(s[nt][2 + e] - mn_b);
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
    // O += P V: 4 k-steps of 16 keys, HD/8 n-tiles of 8 dims.  P is carried as
    // a bf16 pair hi + lo (two MMAs), about 16 significant bits, so the weights
    // are not rounded to 8 bits before they meet V.
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ph[4], pl[4];
      split_bf16x2(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
      split_bf16x2(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
      split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
      split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
      for (int nd = 0; nd < HD / 8; nd += 2) {
        const int mat = lane >> 3;
        const int key = kk * 16 + (mat & 1) * 8 + (lane & 7);
        const int ch = nd + (mat >> 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vs_base + key * ROWB + ((ch ^ (key & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_16816(o[nd], ph, b0, b1);
        mma_bf16_16816(o[nd], pl, b0, b1);
        mma_bf16_16816(o[nd + 1], ph, b2, b3);
        mma_bf16_16816(o[nd + 1], pl, b2, b3);
      }
    }
  }
  cp_async_wait<0>();

  // quad-reduce the row sums and write this split's partials
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int rr = half ? rb : ra;
    if (rr >= rows) continue;
    const size_t idx = (static_cast<size_t>(split) * n_samp + row_sample(rr)) * a.H + row_head(rr);
    float* po = a.part_o + idx * HD;
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd) {
      const int d = nd * 8 + tq * 2;
      *reinterpret_cast<float2*>(po + d) = make_float2(o[nd][half * 2], o[nd][half * 2 + 1]);
    }
    if (tq == 0) {
      a.part_ml[idx * 2] = half ? m_b : m_a;
      a.part_ml[idx * 2 + 1] = half ? l_b : l_a;
    }
  }
}

// out[s][h*hd + d] = sum_j 2^(m_j - M) o_j[d] / sum_j 2^(m_j - M) l_j.
// Warp 0 turns the (m_j, l_j) of the splits into weights once; then every
// thread sums its dimensions over the splits.
template <typename T>
__global__ void attn_combine_kernel(const AttnArgs a) {
  __shared__ float w_sh[kMaxSplits];
  __shared__ float inv_sh;
  pdl_trigger();
  pdl_wait();
  const size_t sh = blockIdx.x;  // (sample, head)
  const size_t n_sh = static_cast<size_t>(a.B) * a.K * a.H;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float M = -INFINITY;
    for (int j = lane; j < a.n_splits; j += 32) M = fmaxf(M, a.part_ml[(j * n_sh + sh) * 2]);
    M = warp_max(M);
    float den = 0.f;
    for (int j = lane; j < a.n_splits; j += 32) {
      const float m = a.part_ml[(j * n_sh + sh) * 2];
      const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
      w_sh[j] = w;
      den += w * a.part_ml[(j * n_sh + sh) * 2 + 1];
    }
    den = warp_sum(den);
    if (lane == 0) inv_sh = den > 0.f ? 1.f / den : 0.f;
  }
  __syncthreads();
  const float inv = inv_sh;
  for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
    // eight independent accumulators keep eight split loads in flight
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int j = 0;
    for (; j + 8 <= a.n_splits; j += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u)
        acc[u] += w_sh[j + u] * a.part_o[((j + u) * n_sh + sh) * a.hd + d];
    }
    for (; j < a.n_splits; ++j) acc[0] += w_sh[j] * a.part_o[(j * n_sh + sh) * a.hd + d];
    const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    static_cast<T*>(a.out)[sh * a.hd + d] = Elem<T>::from_f(sum * inv);
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
  if (L > Lmax || L < a.K) {
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
  float M = -INFINITY;
  for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w]);
  float den = 0.f;
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
                    int& n_splits, int& split_len) {
  (void)K;
  (void)H;
  (void)hd;
  const long Lmax = static_cast<long>(max_blocks) * bs;
  const long chunks = std::max<long>(1, (Lmax + kKC - 1) / kKC);
  const long ns = attention_split_count(B, G, max_blocks, bs, num_sms);
  const long chunks_per = (chunks + ns - 1) / ns;
  split_len = static_cast<int>(chunks_per * kKC);
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
  const int warps = (rows + 15) / 16;
  const dim3 grid(a.n_splits, a.G, a.B);
  const int stages = a.hd >= 128 ? ring_stages<128>() : ring_stages<64>();
  const size_t smem = static_cast<size_t>(stages) * 2 * kKC * a.hd * 2;
  // one attribute value for every launch (the largest ring)
  const int smem_max = 3 * 2 * kKC * 128 * 2;
  if (a.hd == 64) {
    cudaFuncSetAttribute(attn_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (launch_pdl(attn_mma_kernel<64>, grid, dim3(warps * 32), smem, st, a) != cudaSuccess)
      return PE_ERR_CUDA;
  } else if (a.hd == 128) {
    cudaFuncSetAttribute(attn_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (launch_pdl(attn_mma_kernel<128>, grid, dim3(warps * 32), smem, st, a) != cudaSuccess)
      return PE_ERR_CUDA;
  } else {
    return PE_ERR_UNSUPPORTED;
  }
  if (cudaGetLastError() != cudaSuccess) return PE_ERR_CUDA;
  return launch_pdl(attn_combine_kernel<bf16>, dim3(a.B * a.K * a.H), dim3(std::min(a.hd, 128)), 0,
                    st, a) == cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}

}  // namespace pe
