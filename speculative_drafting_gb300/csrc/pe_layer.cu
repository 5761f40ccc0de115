// Row RMSNorm, rotary embedding with the paged KV write, and the argmax
// finalisation of the drafter layer.
//
// RoPE is the rotate-half form: the pair (x_i, x_{i+hd/2}) turns by the angle
// pos * theta^(-2i/hd).  The angle is formed and reduced modulo 2*pi in double
// precision (positions reach 32K and beyond, where a float product would lose
// ~1e-3 rad), then sincosf runs on the reduced angle.
//
// KV write: non-rejected rows store k (after RoPE) and v at their slot; rejected
// rows never reach this kernel (their slot is PADDING_SLOT_ID = -1, "P-EAGLE:
// parallel speculative decoding in vLLM", KV cache and CUDA graphs).
#include "pe_common.cuh"
#include "pe_prep.h"

namespace pe {

template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const T* __restrict__ x, int ld_x,
                                                      const T* __restrict__ gamma,
                                                      T* __restrict__ out, int ld_out, int d,
                                                      float eps, int rows_cap,
                                                      const int* n_rows_dev) {
  __shared__ float red[32];
  constexpr int V = Elem<T>::kVec;
  const int row = blockIdx.x;
  int n = rows_cap;
  if (n_rows_dev) n = min(max(*n_rows_dev, 0), rows_cap);
  if (row >= n) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(row) * ld_x);
  const uint4* gam = reinterpret_cast<const uint4*>(gamma);
  uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(row) * ld_out);
  const int vd = d / V;
  float ss = 0.f;
  for (int i = threadIdx.x; i < vd; i += blockDim.x) {
    float f[V];
    unpack16<T>(src[i], f);
#pragma unroll
    for (int k = 0; k < V; ++k) ss = fmaf(f[k], f[k], ss);
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(d) + eps);
  for (int i = threadIdx.x; i < vd; i += blockDim.x) {
    float f[V], g[V];
    unpack16<T>(src[i], f);
    unpack16<T>(gam[i], g);
#pragma unroll
    for (int k = 0; k < V; ++k) f[k] = f[k] * inv * g[k];
    dst[i] = pack16<T>(f);
  }
}

int launch_rmsnorm(const void* x, int ld_x, const void* gamma, void* out, int ld_out, int d,
                   float eps, int rows_cap, const int* n_rows_dev, int dtype, cudaStream_t st) {
  if (rows_cap <= 0) return PE_OK;
  const int threads = d >= 2048 ? 256 : 128;
  if (dtype == PE_DTYPE_BF16)
    rmsnorm_kernel<bf16><<<rows_cap, threads, 0, st>>>(
        static_cast<const bf16*>(x), ld_x, static_cast<const bf16*>(gamma),
        static_cast<bf16*>(out), ld_out, d, eps, rows_cap, n_rows_dev);
  else
    rmsnorm_kernel<float><<<rows_cap, threads, 0, st>>>(
        static_cast<const float*>(x), ld_x, static_cast<const float*>(gamma),
        static_cast<float*>(out), ld_out, d, eps, rows_cap, n_rows_dev);
  return cudaGetLastError() == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

// ------------------------------------------------------------------ RoPE + KV write

// One CTA per non-rejected row v.  The row is a sample row when it is one of
// the last K non-rejected rows of its request (NTP row + MASK rows).
template <typename T>
__global__ void __launch_bounds__(256) rope_kv_kernel(const RopeArgs a) {
  __shared__ float cs[64], sn[64];
  __shared__ int samp_sh;
  const int v = blockIdx.x;
  const int nv = min(max(*a.n_valid, 0), a.T_out);
  if (v >= nv) return;
  const int o = a.valid_rows[v];
  if (o < 0 || o >= a.T_out) {
    if (threadIdx.x == 0) set_status(a.status, PE_ST_ACCEPTED_RANGE);
    return;
  }
  const int half = a.hd / 2;
  const int64_t p = a.pos[o];
  const int64_t slot = a.slot[o];
  if (threadIdx.x == 0) {
    // request of row v: largest r with valid_qsl[r] <= v
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.valid_qsl[mid] <= v)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int k = v - (a.valid_qsl[lo + 1] - a.K);
    samp_sh = (k >= 0 && k < a.K) ? lo * a.K + k : -1;
  }
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double ang = static_cast<double>(p) * a.inv_freq[i];
    const double two_pi = 6.283185307179586476925286766559;
    const double red = ang - two_pi * rint(ang / two_pi);
    float s, c;
    sincosf(static_cast<float>(red), &s, &c);
    cs[i] = c;
    sn[i] = s;
  }
  __syncthreads();
  const int s_idx = samp_sh;
  const int QKV = (a.H + 2 * a.G) * a.hd;
  const float* row = a.qkv + static_cast<size_t>(v) * QKV;
  const bool slot_ok = slot >= 0 && slot < static_cast<int64_t>(a.num_blocks) * a.bs;
  if (!slot_ok && slot != PE_PADDING_SLOT_ID && threadIdx.x == 0)
    set_status(a.status, PE_ST_BLOCK_RANGE);
  const int64_t blk = slot_ok ? slot / a.bs : 0, off = slot_ok ? slot % a.bs : 0;
  // rotated q (sample rows) and k (all rows)
  for (int e = threadIdx.x; e < (a.H + a.G) * half; e += blockDim.x) {
    const int hh = e / half, i = e - hh * half;
    const float x1 = row[hh * a.hd + i], x2 = row[hh * a.hd + i + half];
    const float y1 = x1 * cs[i] - x2 * sn[i];
    const float y2 = x2 * cs[i] + x1 * sn[i];
    if (hh < a.H) {
      if (s_idx < 0) continue;
      T* q = static_cast<T*>(a.q_s) + (static_cast<size_t>(s_idx) * a.H + hh) * a.hd;
      q[i] = Elem<T>::from_f(y1);
      q[i + half] = Elem<T>::from_f(y2);
    } else if (slot_ok) {
      const int g = hh - a.H;
      T* kc = static_cast<T*>(a.k_cache) + ((blk * a.G + g) * a.bs + off) * a.hd;
      kc[i] = Elem<T>::from_f(y1);
      kc[i + half] = Elem<T>::from_f(y2);
    }
  }
  if (slot_ok) {
    for (int e = threadIdx.x; e < a.G * a.hd; e += blockDim.x) {
      const int g = e / a.hd, i = e - g * a.hd;
      T* vc = static_cast<T*>(a.v_cache) + ((blk * a.G + g) * a.bs + off) * a.hd;
      vc[i] = Elem<T>::from_f(row[(a.H + a.G) * a.hd + e]);
    }
  }
  if (s_idx >= 0) {
    constexpr int V = Elem<T>::kVec;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) +
                                                      static_cast<size_t>(v) * a.d);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(a.x_s) + static_cast<size_t>(s_idx) * a.d);
    for (int i = threadIdx.x; i < a.d / V; i += blockDim.x) dst[i] = src[i];
  }
}

int launch_rope_kv(const RopeArgs& a, int dtype, cudaStream_t st) {
  if (a.T_out <= 0) return PE_OK;
  if (dtype == PE_DTYPE_BF16)
    rope_kv_kernel<bf16><<<a.T_out, 256, 0, st>>>(a);
  else
    rope_kv_kernel<float><<<a.T_out, 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

// ------------------------------------------------------------------ argmax keys -> ids

__global__ void argmax_finalize_kernel(const unsigned long long* __restrict__ keys, int n,
                                       int32_t* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const unsigned long long k = keys[i];
  out[i] = k ? static_cast<int32_t>(~static_cast<uint32_t>(k & 0xffffffffull)) : 0;
}

int launch_argmax_finalize(const unsigned long long* keys, int n, int32_t* out, cudaStream_t st) {
  if (n <= 0) return PE_OK;
  argmax_finalize_kernel<<<(n + 255) / 256, 256, 0, st>>>(keys, n, out);
  return cudaGetLastError() == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

}  // namespace pe
