// Greedy verification of a ragged verify batch: the target's greedy token of
// every verify row, each request's accepted-draft count and its bonus token.
//
// "Attention Drift", section 2 (preliminaries): the target scores the drafted
// tokens in one forward pass and keeps the longest prefix it accepts.  The
// drafts of the parallel-draft step are greedy, so acceptance here is exact
// agreement with the target's greedy token (temperature 0).  The results are the
// accepted counts and bonus tokens that the next pe_prepare_inputs takes.
//
// Two kernels, chained by programmatic launch:
//   verify_partial_kernel  streams the logits once.  CTA (row, s) scans a chunk
//                          of one row with 16-byte loads (a scalar head up to the
//                          first 16-byte boundary and a scalar tail), compares
//                          only each vector's NaN-propagating maximum, keeps
//                          the first vector that holds the best value in
//                          registers, finds its lowest index holding the value
//                          at the end, and writes the chunk's (value, lowest
//                          index) key.
//                          HBM-bound.
//   verify_accept_kernel   one CTA per request: each row's target token is the
//                          largest of its chunk keys; the first draft that
//                          differs from the pick of the row before it ends the
//                          accepted prefix.
#include <algorithm>

#include "pe_common.cuh"
#include "pe_internal.h"

namespace pe {
namespace {

constexpr int kPartThreads = 256;
constexpr int kAcceptThreads = 128;
constexpr int kUnroll = 4;          // 16-byte loads in flight per thread
constexpr int kMaxChunkBytes = 32768;
constexpr int kWsHeader = 256;      // status word, then the chunk keys

PE_DEV uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <typename T>
PE_DEV float elem_f(const T* p);
template <>
PE_DEV float elem_f<float>(const float* p) { return *p; }
template <>
PE_DEV float elem_f<bf16>(const bf16* p) { return __bfloat162float(*p); }

// Keep the greater of (bk, bi) and (order of v, idx).  A thread visits its
// elements in increasing index order, so the strict comparison keeps the lowest
// index among equal values.
PE_DEV void consider(float v, uint32_t idx, uint32_t& bk, uint32_t& bi) {
  const uint32_t k = argmax_order(v);
  if (k > bk) {
    bk = k;
    bi = idx;
  }
}

PE_DEV float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

PE_DEV uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest element of a 16-byte vector, NaN if it holds one.
template <typename T>
PE_DEV float vec_max(const uint4& u);
template <>
PE_DEV float vec_max<float>(const uint4& u) {
  return max_nan(max_nan(__uint_as_float(u.x), __uint_as_float(u.y)),
                 max_nan(__uint_as_float(u.z), __uint_as_float(u.w)));
}
template <>
PE_DEV float vec_max<bf16>(const uint4& u) {
  // pairwise on packed bf16 pairs, then the two halves (bf16 -> fp32 is exact)
  const uint32_t p = max_nan_bf16x2(max_nan_bf16x2(u.x, u.y), max_nan_bf16x2(u.z, u.w));
  return max_nan(__uint_as_float(p << 16), __uint_as_float(p & 0xffff0000u));
}

template <typename T>
__global__ void __launch_bounds__(kPartThreads, 6) verify_partial_kernel(
    const T* __restrict__ logits, int V, int chunk, int splits,
    unsigned long long* __restrict__ part, uint32_t* status) {
  constexpr int kVec = 16 / sizeof(T);
  __shared__ unsigned long long wmax[kPartThreads / 32];
  pdl_trigger();
  pdl_wait();  // the logits may come from the previous kernel on the stream
  const int row = blockIdx.x / splits, s = blockIdx.x - row * splits, tid = threadIdx.x;
  // only the accept kernel, which runs after this one, sets status bits
  if (blockIdx.x == 0 && tid == 0) *status = 0u;
  const int c0 = s * chunk, c1 = min(V, c0 + chunk);
  const T* base = logits + static_cast<size_t>(row) * static_cast<size_t>(V);
  // every real value orders above 0, so an idle thread's (0, -) loses
  uint32_t bk = 0u, bi = 0xffffffffu;
  // scalar head: up to the first 16-byte boundary at or after element c0
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(base + c0);
  const int head = min(static_cast<int>(((16u - (a0 & 15u)) & 15u) / sizeof(T)), c1 - c0);
  if (tid < head) consider(elem_f(base + c0 + tid), static_cast<uint32_t>(c0 + tid), bk, bi);
  const int v0 = c0 + head;
  const int nvec = (c1 - v0) / kVec;
  const uint4* vp = reinterpret_cast<const uint4*>(base + v0);
  // Vector pass: each 16-byte vector is reduced to its maximum (NaN if it holds
  // one) and the thread keeps, without branching, the first vector (in its
  // increasing index order) whose maximum is its greatest value so far -- a NaN
  // counts as the greatest, and once the best is a NaN nothing replaces it.
  // The kept vector's bits stay in registers; after the loop its lowest index
  // that holds the value is found.
  float best = 0.f;
  int bj = -1;
  uint4 bv = make_uint4(0u, 0u, 0u, 0u);
  for (int j = tid; j < nvec; j += kUnroll * kPartThreads) {
    uint4 u[kUnroll];
#pragma unroll
    for (int x = 0; x < kUnroll; ++x)
      if (j + x * kPartThreads < nvec) u[x] = ld_stream16(vp + j + x * kPartThreads);
#pragma unroll
    for (int x = 0; x < kUnroll; ++x) {
      if (j + x * kPartThreads < nvec) {
        const float m = vec_max<T>(u[x]);
        const bool upd = bj < 0 || (!(m <= best) && best == best);
        best = upd ? m : best;
        bj = upd ? j + x * kPartThreads : bj;
        bv.x = upd ? u[x].x : bv.x;
        bv.y = upd ? u[x].y : bv.y;
        bv.z = upd ? u[x].z : bv.z;
        bv.w = upd ? u[x].w : bv.w;
      }
    }
  }
  if (bj >= 0) {
    float f[kVec];
    unpack16<T>(bv, f);
    int e = kVec - 1;
#pragma unroll
    for (int i = kVec - 1; i >= 0; --i)
      if (best != best ? f[i] != f[i] : f[i] == best) e = i;
    consider(best, static_cast<uint32_t>(v0 + bj * kVec + e), bk, bi);
  }
  // scalar tail
  const int t0 = v0 + nvec * kVec;
  if (t0 + tid < c1) consider(elem_f(base + t0 + tid), static_cast<uint32_t>(t0 + tid), bk, bi);

  // consider() kept the greater of the head, the vector pass and the tail, in
  // index order, so ties among them also go to the lowest index
  unsigned long long key =
      (static_cast<unsigned long long>(bk) << 32) | static_cast<unsigned long long>(~bi);
  key = warp_max_u64(key);
  if ((tid & 31) == 0) wmax[tid >> 5] = key;
  __syncthreads();
  if (tid < 32) {
    key = tid < kPartThreads / 32 ? wmax[tid] : 0ull;
    key = warp_max_u64(key);
    if (tid == 0) part[static_cast<size_t>(row) * splits + s] = key;
  }
}

__global__ void __launch_bounds__(kAcceptThreads) verify_accept_kernel(
    int B, int T_in, int splits, const int32_t* __restrict__ qsl, const int32_t* __restrict__ tok,
    const unsigned long long* __restrict__ part, int32_t* __restrict__ target_tok,
    int32_t* __restrict__ accepted, int32_t* __restrict__ bonus, uint32_t* status) {
  __shared__ int first_bad;
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();
  int q0 = qsl[r], q1 = qsl[r + 1];
  bool bad = q0 < 0 || q1 > T_in || q1 < q0 || (r == 0 && q0 != 0) || (r == B - 1 && q1 != T_in);
  q0 = min(max(q0, 0), T_in);
  q1 = min(max(q1, q0), T_in);
  if (bad && tid == 0) set_status(status, PE_ST_ROWS_RANGE);
  const int n = q1 - q0;
  if (tid == 0) first_bad = n;
  __syncthreads();
  // one warp per row: the row's target token is the largest of its chunk keys
  for (int j = warp; j < n; j += kAcceptThreads / 32) {
    const unsigned long long* pk = part + static_cast<size_t>(q0 + j) * splits;
    unsigned long long k = 0ull;
    for (int s = lane; s < splits; s += 32) k = max(k, pk[s]);
    k = warp_max_u64(k);
    const int32_t t = static_cast<int32_t>(~static_cast<uint32_t>(k));
    if (lane == 0) {
      target_tok[q0 + j] = t;
      // draft j+1 follows row j: it is accepted only if it is the target's pick
      if (j + 1 < n && tok[q0 + j + 1] != t) atomicMin(&first_bad, j);
    }
  }
  __syncthreads();  // also makes this CTA's target_tok stores visible to thread 0
  if (tid == 0) {
    const int a = n > 0 ? min(first_bad, n - 1) : 0;
    accepted[r] = a;
    bonus[r] = n > 0 ? target_tok[q0 + a] : -1;
  }
}

struct VerifyPlan {
  int chunk, splits;
};

// Chunk of a row per CTA: about one wave of CTAs (six per SM) over the whole
// batch, between one 16-byte vector per thread and 32 KB, a whole number of
// vectors.  (8 rows of 201,088 fp32 logits: 12.1 us against 12.8-14.1 us with
// sixteen CTAs per SM; large batches are capped by the 32 KB chunk either way.)  (Measured on
// 512 rows of 201,088 bf16 logits: 43 us with 32 KB chunks, 45 us with 64 KB,
// 48-50 us with 128 KB; fp32 logits 73.5 us with 32 or 64 KB.)
VerifyPlan plan_verify(int T_in, int V, int esize, int num_sms) {
  const int vec = 16 / esize;
  const long long total = static_cast<long long>(T_in) * V;
  const long long target_ctas = 6LL * num_sms;
  long long chunk = (total + target_ctas - 1) / target_ctas;
  chunk = std::max<long long>(chunk, static_cast<long long>(kPartThreads) * vec);
  chunk = std::min<long long>(chunk, kMaxChunkBytes / esize);
  chunk = (chunk + vec - 1) / vec * vec;
  VerifyPlan p;
  p.chunk = static_cast<int>(chunk);
  p.splits = static_cast<int>((V + chunk - 1) / chunk);
  return p;
}

// the most chunk keys a row can need (the smallest chunk: fp32, one vector per thread)
long long max_splits(int V) {
  const long long min_chunk = static_cast<long long>(kPartThreads) * 4;
  return (V + min_chunk - 1) / min_chunk;
}

}  // namespace
}  // namespace pe

using namespace pe;

extern "C" size_t pe_verify_workspace_bytes(int max_rows_in, int vocab) {
  if (max_rows_in < 0 || vocab < 1) return 0;
  const size_t keys = static_cast<size_t>(max_rows_in) * static_cast<size_t>(max_splits(vocab));
  return static_cast<size_t>(kWsHeader) + keys * sizeof(unsigned long long);
}

extern "C" int pe_verify_greedy(int B, int T_in, const int32_t* qsl, const int32_t* tok,
                                const void* logits, int vocab, int dtype, int32_t* target_tok,
                                int32_t* accepted, int32_t* bonus, void* ws, size_t ws_bytes,
                                void* stream) {
  NvtxRange nvtx("pe_verify_greedy");
  if (B < 0 || T_in < 0 || vocab < 1) return PE_ERR_ARG;
  if (dtype != PE_DTYPE_F32 && dtype != PE_DTYPE_BF16) return PE_ERR_UNSUPPORTED;
  if (B == 0) return T_in == 0 ? PE_OK : PE_ERR_ARG;
  if (!qsl || !accepted || !bonus || !ws) return PE_ERR_ARG;
  if (T_in > 0 && (!tok || !logits || !target_tok)) return PE_ERR_ARG;
  const int esize = dtype == PE_DTYPE_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(logits) % esize != 0) return PE_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return PE_ERR_ARG;
  if (ws_bytes < pe_verify_workspace_bytes(T_in, vocab)) return PE_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t* status = static_cast<uint32_t*>(ws);
  unsigned long long* part = reinterpret_cast<unsigned long long*>(
      static_cast<char*>(ws) + kWsHeader);
  const VerifyPlan p = plan_verify(T_in, vocab, esize, num_sms_of_current_device());
  if (static_cast<long long>(T_in) * p.splits > 0x7fffffffLL) return PE_ERR_UNSUPPORTED;
  if (T_in > 0) {
    // one CTA per (row, chunk); the first also clears the status word
    const dim3 grid(T_in * p.splits);
    const cudaError_t e =
        dtype == PE_DTYPE_F32
            ? launch_pdl(verify_partial_kernel<float>, grid, dim3(kPartThreads), 0, st,
                         static_cast<const float*>(logits), vocab, p.chunk, p.splits, part,
                         status)
            : launch_pdl(verify_partial_kernel<bf16>, grid, dim3(kPartThreads), 0, st,
                         static_cast<const bf16*>(logits), vocab, p.chunk, p.splits, part,
                         status);
    if (e != cudaSuccess) return PE_ERR_CUDA;
  } else if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) {
    return PE_ERR_CUDA;
  }
  return launch_pdl(verify_accept_kernel, dim3(B), dim3(kAcceptThreads), 0, st, B, T_in,
                    p.splits, qsl, tok, static_cast<const unsigned long long*>(part), target_tok,
                    accepted, bonus, status) == cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}
