// The asymmetric attention mask of COD training, from the index lists.
//
// "[RFC]: Add random anchor for p-eagle first position", Proposed change: the
// mask's queries are the COD tokens, its keys the whole sequence plus the deeper
// COD tokens; the reply's "Depth > 0 attention": a deeper query sees the
// sequence up to its anchor as well as its own chain.
//
//   cod_mask_kernel   one warp per query row (anchor a, depth k): columns 0..a of
//                     the original sequence and the row's own chain columns at
//                     depths 1..k are 1, every other column below the row's key
//                     count 0, written with 16-byte stores.  Bound by the mask's
//                     bytes (HBM).
#include "pe_cod_internal.h"

namespace pe {
namespace {

// Row q of sequence b (depth-major): anchor a, depth k.  The mask row holds the
// key columns 0..KV-1 (the L original positions, then the depth >= 1 tokens in
// depth-major order) and is written up to the next multiple of 16 bytes.
__global__ void __launch_bounds__(kMaskThreads) cod_mask_kernel(
    int S_max, const int32_t* __restrict__ seq_len, int D, const int32_t* __restrict__ idx,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ place, uint8_t* __restrict__ mask,
    long long q_cap, long long ld, long long mstride, uint32_t* status) {
  __shared__ int qoff[kMaxD + 1];
  __shared__ int spc[kMaskWarps][kMaxD];
  const int b = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_trigger();
  pdl_wait();
  const int L_in = seq_len[b];
  const int L = clamp_len(L_in, S_max);
  if (threadIdx.x == 0) {
    uint32_t bad = L != L_in ? PE_ST_CAPACITY : 0u;
    int s = 0;
    for (int k = 0; k < D; ++k) {
      int n = counts[b * D + k];
      if (n < 0 || n > L) {
        bad |= PE_ST_CAPACITY;
        n = n < 0 ? 0 : L;
      }
      qoff[k] = s;
      s += n;
    }
    qoff[D] = s;
    if (bad && blockIdx.x == 0) set_status(status, bad);
  }
  __syncthreads();
  const long long Q = qoff[D];
  const long long n0 = qoff[1];
  const long long KV = L + Q - n0;
  long long rows = Q, width = (KV + 15) / 16 * 16;
  if (rows > q_cap || width > ld) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, PE_ST_CAPACITY);
    rows = rows < q_cap ? rows : q_cap;
    width = width < ld ? width : ld;
  }
  uint8_t* mb = mask + static_cast<long long>(b) * mstride;
  const int32_t* ib = idx + static_cast<size_t>(b) * D * S_max;
  const int32_t* pb = D > 1 ? place + static_cast<size_t>(b) * (D - 1) * S_max : nullptr;
  const long long nvec = width / 16;
  const long long stride = static_cast<long long>(gridDim.x) * kMaskWarps;
  // row q's anchor (and its depth) is loaded one row ahead, so its latency
  // overlaps the previous row's stores
  auto anchor_of = [&](long long q, int& k) {
    k = 0;
    while (k + 1 < D && qoff[k + 1] <= q) ++k;
    return ib[static_cast<size_t>(k) * S_max + (q - qoff[k])];
  };
  long long q = static_cast<long long>(blockIdx.x) * kMaskWarps + warp;
  int k_next = 0;
  int a_next = q < rows ? anchor_of(q, k_next) : 0;
  for (; q < rows; q += stride) {
    const int k = k_next, a = a_next;
    if (q + stride < rows) a_next = anchor_of(q + stride, k_next);
    if (a < 0 || a >= L) {  // not a list this kernel's sibling wrote
      if (lane == 0) set_status(status, PE_ST_CAPACITY);
      continue;
    }
    // the row's own chain token at depth j (1..k) is key column
    // L + (qoff[j] - n0) + its place in depth j's list
    if (lane >= 1 && lane <= k) {
      const int p = pb[static_cast<size_t>(lane - 1) * S_max + a];
      const bool ok = p >= 0 && p < qoff[lane + 1] - qoff[lane];
      if (!ok) set_status(status, PE_ST_CAPACITY);
      spc[warp][lane] = ok ? static_cast<int>(L + (qoff[lane] - n0) + p) : -1;
    }
    __syncwarp();
    uint8_t* rowp = mb + q * ld;
    for (long long v = lane; v < nvec; v += 32) {
      const long long c0 = v * 16;
      uint32_t w[4];
      if (c0 + 15 <= a) {  // wholly inside the context the row sees
        w[0] = w[1] = w[2] = w[3] = 0x01010101u;
      } else {
        w[0] = w[1] = w[2] = w[3] = 0u;
        if (c0 <= a) {  // the one vector that holds column a
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint32_t x = 0;
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (c0 + 4 * h + t <= a) x |= 1u << (8 * t);
            w[h] = x;
          }
        }
        if (c0 + 16 > L) {  // reaches the chain tokens' columns
          for (int j = 1; j <= k; ++j) {
            const long long s = spc[warp][j] - c0;
            if (s >= 0 && s < 16) w[s >> 2] |= 1u << (8 * (s & 3));
          }
        }
      }
      *reinterpret_cast<uint4*>(rowp + c0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncwarp();
  }
}

}  // namespace
}  // namespace pe

using namespace pe;

extern "C" int pe_cod_mask(int B, int S_max, const int32_t* seq_len, int n_depth,
                           const int32_t* idx, const int32_t* counts, uint8_t* mask, int64_t q_cap,
                           int64_t ld, int64_t mask_stride, void* ws, size_t ws_bytes,
                           void* stream) {
  NvtxRange nvtx("pe_cod_mask");
  const int e = cod_common_args(B, S_max, n_depth, seq_len, ws, ws_bytes);
  if (e != PE_OK) return e;
  if (q_cap < 0 || ld < 16 || ld % 16 != 0 || mask_stride % 16 != 0) return PE_ERR_ARG;
  if (q_cap > INT64_MAX / ld || (q_cap > 0 && mask_stride < q_cap * ld)) return PE_ERR_ARG;
  if (B > 0 && (!counts || !idx || !mask)) return PE_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(mask) % 16 != 0) return PE_ERR_ARG;
  if (B == 0 || q_cap == 0) return PE_OK;
  const int sms = num_sms_of_current_device();
  const int gx = (4 * sms + B - 1) / B;
  const int32_t* place = reinterpret_cast<const int32_t*>(static_cast<const char*>(ws) + kWsHeader);
  return launch_pdl(cod_mask_kernel, dim3(gx < 1 ? 1 : gx, B), dim3(kMaskThreads), 0,
                    static_cast<cudaStream_t>(stream), S_max, seq_len, n_depth, idx, counts, place,
                    mask, static_cast<long long>(q_cap), static_cast<long long>(ld),
                    static_cast<long long>(mask_stride), static_cast<uint32_t*>(ws)) == cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}
