// COD training indices (the mask built on them is in pe_cod_mask.cu).
//
// "[RFC]: Add random anchor for p-eagle first position": COD sampling starts a
// chain at every loss position (with max_anchors, at a uniform random subset of
// them) and keeps a share of each depth's chains for the next depth; the mask's
// queries are the COD tokens, its keys the original sequence plus the deeper COD
// tokens.  The reply's "Depth > 0 attention": a deeper query sees the original
// sequence (up to its anchor), not only its own chain.
//
// The index call's kernel (the mask call's kernel follows it by programmatic
// launch):
//   cod_index_kernel  one CTA per sequence.  Counts the loss positions; when the
//                     cap binds, a three-pass radix select (11 + 11 + 10 bits)
//                     over the candidates' random keys finds the cap-th
//                     smallest (u, position) key.  One pass over the positions,
//                     1024 at a time, then walks each chain's draws to its depth
//                     and writes every depth's list with one ballot and one warp
//                     scan per depth, plus each chain member's place in its
//                     depth's list (the mask kernel's column lookup).
//                     Latency-bound.
#include "pe_cod_internal.h"

namespace pe {
namespace {

constexpr int kIdxThreads = 1024;
constexpr int kIdxWarps = kIdxThreads / 32;

PE_DEV int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// place[b][k-1][a] = index of anchor a in depth k's list (k >= 1; written for
// chain members only).  counts[b][k] = |I_k|; idx[b][k][j] = I_k[j], ascending.
// MAXD >= D bounds the unrolled per-depth loops.
template <int MAXD>
__global__ void __launch_bounds__(kIdxThreads) cod_index_kernel(
    int S_max, const int32_t* __restrict__ seq_len, const uint8_t* __restrict__ loss_mask, int D,
    float rho, int A, const float* __restrict__ u_anchor, const float* __restrict__ u_keep,
    int32_t* __restrict__ idx, int32_t* __restrict__ counts, int32_t* __restrict__ place,
    uint32_t* status) {
  __shared__ int hist[2048];
  __shared__ int red[kIdxWarps];
  __shared__ int wofs[MAXD][kIdxWarps];
  __shared__ int base[MAXD];
  __shared__ int tot[MAXD];
  __shared__ int pick[2];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();
  const int L_in = seq_len[b];
  const int L = clamp_len(L_in, S_max);
  if (L != L_in && tid == 0) set_status(status, PE_ST_CAPACITY);
  const size_t row = static_cast<size_t>(b) * S_max;
  const uint8_t* lm = loss_mask + row;
  const uint32_t* ua = reinterpret_cast<const uint32_t*>(u_anchor) + row;
  const float* uk = D > 1 ? u_keep + static_cast<size_t>(b) * (D - 1) * S_max : nullptr;

  // ---- depth 0: the anchors.  With a binding cap, the cap smallest keys
  // (u bits, position) among the loss positions; u >= 0, so the bits order as
  // the values.
  bool capped = false;
  uint32_t thr = 0;
  int need_eq = 0;  // keys equal to thr taken, lowest positions first
  if (A > 0) {
    int c = 0;
#pragma unroll 4
    for (int i = tid; i < L; i += kIdxThreads) c += lm[i] != 0;
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) red[warp] = c;
    __syncthreads();
    int n = 0;
    for (int w = 0; w < kIdxWarps; ++w) n += red[w];
    capped = n > A;
    if (capped) {
      uint32_t prefix = 0, pmask = 0;
      int rank = A;  // 1-based rank of the wanted key among those matching prefix
      for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int nb = pass == 2 ? 1024 : 2048;
        for (int j = tid; j < nb; j += kIdxThreads) hist[j] = 0;
        __syncthreads();
#pragma unroll 4
        for (int i = tid; i < L; i += kIdxThreads) {
          // both loads issue together (the key does not wait for the mask byte)
          const uint8_t m = lm[i];
          const uint32_t k = ua[i];
          if (m && (k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & (nb - 1)], 1);
        }
        __syncthreads();
        if (warp == 0) {
          // lane l sums bins [l*per, (l+1)*per); the lane whose range holds the
          // rank walks its bins
          const int per = nb / 32;
          int s = 0;
          for (int j = 0; j < per; ++j) s += hist[lane * per + j];
          const int inc = warp_inclusive_scan(s);
          const int exc = inc - s;
          if (exc < rank && rank <= inc) {
            int r = rank - exc, d = lane * per;
            const int end = d + per - 1;
            while (d < end && hist[d] < r) {
              r -= hist[d];
              ++d;
            }
            pick[0] = d;
            pick[1] = r;
          }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(pick[0]) << shift;
        pmask |= static_cast<uint32_t>(nb - 1) << shift;
        rank = pick[1];
        __syncthreads();
      }
      thr = prefix;
      need_eq = rank;
    }
  }

  // ---- every depth's list, 1024 positions at a time
  if (tid < MAXD) base[tid] = 0;
  __syncthreads();
  int eq_seen = 0;  // keys equal to thr met so far (same on every thread)
  for (int c0 = 0; c0 < L; c0 += kIdxThreads) {
    const int i = c0 + tid;
    // the position's mask byte, key and chain draws are loaded together: one
    // memory latency per chunk
    const bool in = i < L;
    const uint8_t m = in ? lm[i] : 0;
    const uint32_t key = (capped && in) ? ua[i] : 0u;
    float uu[MAXD > 1 ? MAXD - 1 : 1];
#pragma unroll
    for (int k = 0; k < MAXD - 1; ++k)
      uu[k] = (k < D - 1 && i + k + 1 < L) ? uk[static_cast<size_t>(k) * S_max + i] : 0.f;
    const bool cand = m != 0;
    bool sel = cand;
    if (capped) {
      const uint32_t k = cand ? key : 0u;
      const bool eq = cand && k == thr;
      const unsigned be = __ballot_sync(0xffffffffu, eq);
      if (lane == 0) red[warp] = __popc(be);
      __syncthreads();
      // equal keys in the warps before this one, and in the whole chunk
      const int wv = red[lane];
      const int winc = warp_inclusive_scan(wv);
      const int before = eq_seen + __shfl_sync(0xffffffffu, winc - wv, warp) +
                         __popc(be & ((1u << lane) - 1u));
      const int all = __shfl_sync(0xffffffffu, winc, 31);
      sel = cand && (k < thr || (eq && before < need_eq));
      eq_seen += all;
      __syncthreads();
    }
    // the chain's depth: each further depth needs its draw below rho and its
    // position a + k inside the sequence
    int len = 0;
    if (sel) {
      len = 1;
#pragma unroll
      for (int k = 0; k < MAXD - 1; ++k)
        if (len == k + 1 && k < D - 1 && i + k + 1 < L && uu[k] < rho) len = k + 2;
    }
#pragma unroll
    for (int k = 0; k < MAXD; ++k) {
      const unsigned bk = __ballot_sync(0xffffffffu, len > k);
      if (k < D && lane == 0) wofs[k][warp] = __popc(bk);
    }
    __syncthreads();
    if (warp < D) {
      const int v = wofs[warp][lane];
      const int inc = warp_inclusive_scan(v);
      wofs[warp][lane] = inc - v;
      if (lane == 31) tot[warp] = inc;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < MAXD; ++k) {
      const unsigned bk = __ballot_sync(0xffffffffu, len > k);
      if (k < D && len > k) {
        const int pos = base[k] + wofs[k][warp] + __popc(bk & ((1u << lane) - 1u));
        idx[(static_cast<size_t>(b) * D + k) * S_max + pos] = i;
        if (k > 0) place[(static_cast<size_t>(b) * (D - 1) + (k - 1)) * S_max + i] = pos;
      }
    }
    __syncthreads();
    if (tid < D) base[tid] += tot[tid];
    __syncthreads();
  }
  if (tid < D) counts[b * D + tid] = base[tid];
}

}  // namespace
}  // namespace pe

using namespace pe;

int cod_common_args(int B, int S_max, int n_depth, const void* seq_len, void* ws,
                           size_t ws_bytes) {
  if (B < 0 || S_max < 0 || n_depth < 1 || n_depth > PE_COD_MAX_DEPTH) return PE_ERR_ARG;
  if (B > 65535) return PE_ERR_UNSUPPORTED;
  if (!ws || reinterpret_cast<uintptr_t>(ws) % 256 != 0) return PE_ERR_ARG;
  if (ws_bytes < pe_cod_workspace_bytes(B, S_max, n_depth)) return PE_ERR_ARG;
  if (B > 0 && !seq_len) return PE_ERR_ARG;
  return PE_OK;
}


extern "C" size_t pe_cod_workspace_bytes(int B, int S_max, int n_depth) {
  if (B < 0 || S_max < 0 || n_depth < 1 || n_depth > PE_COD_MAX_DEPTH) return 0;
  return static_cast<size_t>(kWsHeader) +
         static_cast<size_t>(B) * static_cast<size_t>(n_depth - 1) * static_cast<size_t>(S_max) *
             sizeof(int32_t);
}

extern "C" int pe_cod_sample_indices(int B, int S_max, const int32_t* seq_len,
                                     const uint8_t* loss_mask, int n_depth, float retain,
                                     int max_anchors, const float* u_anchor, const float* u_keep,
                                     int32_t* idx, int32_t* counts, void* ws, size_t ws_bytes,
                                     void* stream) {
  NvtxRange nvtx("pe_cod_sample_indices");
  const int e = cod_common_args(B, S_max, n_depth, seq_len, ws, ws_bytes);
  if (e != PE_OK) return e;
  if (!(retain == retain) || max_anchors < 0) return PE_ERR_ARG;
  if (B > 0 && (!counts || (S_max > 0 && (!loss_mask || !u_anchor || !idx ||
                                          (n_depth > 1 && !u_keep)))))
    return PE_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(u_anchor) % 4 != 0 || reinterpret_cast<uintptr_t>(u_keep) % 4 != 0)
    return PE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = static_cast<uint32_t*>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) return PE_ERR_CUDA;
  if (B == 0) return PE_OK;
  int32_t* place = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kWsHeader);
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, dim3(B), dim3(kIdxThreads), 0, st, S_max, seq_len, loss_mask,
                      n_depth, retain, max_anchors, u_anchor, u_keep, idx, counts, place, status);
  };
  const cudaError_t err = n_depth <= 4   ? go(cod_index_kernel<4>)
                          : n_depth <= 8 ? go(cod_index_kernel<8>)
                                         : go(cod_index_kernel<kMaxD>);
  return err == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}
