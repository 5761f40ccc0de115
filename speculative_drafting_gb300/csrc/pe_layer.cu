// Row RMSNorm (fp32 rows in; bf16, bf16-pair or fp32 out), rotary embedding
// with the paged KV write, and the argmax finalisation of the drafter layer.
//
// RoPE is the rotate-half form: the pair (x_i, x_{i+hd/2}) turns by the angle
// pos * theta^(-2i/hd).  The angle is formed and reduced modulo 2*pi in double
// precision (positions reach 32K and beyond, where a float product would lose
// ~1e-3 rad), then sincosf runs on the reduced angle.
//
// KV write: non-rejected rows store k (after RoPE) and v at their slot; rejected
// rows never reach this kernel (their slot is PADDING_SLOT_ID = -1, "P-EAGLE:
// parallel speculative decoding in vLLM", KV cache and CUDA graphs).
#include <algorithm>

#include "pe_common.cuh"
#include "pe_prep.h"

namespace pe {

// One CTA per row: x = (sum of the partial tiles, in order) + resid, then
// y = x * gamma / sqrt(mean(x^2) + eps) (or y = x when apply_norm is 0), stored
// as any of: the step's element type (out, rounded to nearest), the rest of a
// bf16 pair (out_lo = bf16(y - out)), and the fp32 value of what was stored
// (out + out_lo, or y); sum_out receives x.  The row stays in registers between
// the sum of squares and the output pass (up to kRowCache float4 per thread).
constexpr int kRowCache = 4;

template <typename T>
PE_DEV void load_gain4(const T* g, int i, float* out) {
#pragma unroll
  for (int k = 0; k < 4; ++k) out[k] = Elem<T>::to_f(g[4 * i + k]);
}
template <>
PE_DEV void load_gain4<bf16>(const bf16* g, int i, float* out) {
  const uint2 u = reinterpret_cast<const uint2*>(g)[i];  // four bf16 in 8 bytes
  out[0] = __uint_as_float(u.x << 16);
  out[1] = __uint_as_float(u.x & 0xffff0000u);
  out[2] = __uint_as_float(u.y << 16);
  out[3] = __uint_as_float(u.y & 0xffff0000u);
}

// two 16-bit values as one word (the first in the low half)
PE_DEV uint32_t pack2(bf16 a, bf16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// four consecutive values (rounded to T) with one store: 8 bytes for bf16,
// 16 for fp32
template <typename T>
PE_DEV void store4(T* p, const float* v);
template <>
PE_DEV void store4<bf16>(bf16* p, const float* v) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack2(__float2bfloat16_rn(v[0]), __float2bfloat16_rn(v[1])),
                                            pack2(__float2bfloat16_rn(v[2]), __float2bfloat16_rn(v[3])));
}
template <>
PE_DEV void store4<float>(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

template <typename T>
__global__ void __launch_bounds__(256) rownorm_kernel(RowNormArgs a) {
  __shared__ float red[32];
  pdl_trigger();
  const int v4 = a.d / 4;
  // the gains are weights, independent of the kernels before: read them now
  const T* gam = static_cast<const T*>(a.gamma);
  float gc[kRowCache][4];
#pragma unroll
  for (int c = 0; c < kRowCache; ++c) {
    const int i = threadIdx.x + c * blockDim.x;
    if (a.apply_norm && i < v4) {
      load_gain4<T>(gam, i, gc[c]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) gc[c][k] = 1.f;
    }
  }
  pdl_wait();
  const int row = blockIdx.x;
  int n = a.rows_cap;
  if (a.n_rows_dev) n = min(max(*a.n_rows_dev, 0), a.rows_cap);
  if (row >= n) return;
  // input row: the same, or the row-th sample row of a right-aligned layout
  const int irow = a.in_group > 0 ? (row / a.out_group) * a.in_group +
                                        (a.in_group - a.out_group) + row % a.out_group
                                  : row;
  const size_t ro = static_cast<size_t>(irow) * a.ld_x;
  const float4* x0 = reinterpret_cast<const float4*>(a.x + ro);
  const float4* res =
      a.resid ? reinterpret_cast<const float4*>(a.resid + static_cast<size_t>(irow) * a.ld_resid)
              : nullptr;
  auto load = [&](int i) {
    float4 s = x0[i];
    for (int k = 1; k < a.n_parts; ++k) {
      const float4 p = reinterpret_cast<const float4*>(a.x + k * a.part_stride + ro)[i];
      s.x += p.x;
      s.y += p.y;
      s.z += p.z;
      s.w += p.w;
    }
    if (res) {
      const float4 r = res[i];
      s.x += r.x;
      s.y += r.y;
      s.z += r.z;
      s.w += r.w;
    }
    if (a.sum_out) reinterpret_cast<float4*>(a.sum_out + ro)[i] = s;
    return s;
  };
  float4 xc[kRowCache];
  float ss = 0.f;
  auto acc_ss = [&](const float4& f) {
    ss = fmaf(f.x, f.x, ss);
    ss = fmaf(f.y, f.y, ss);
    ss = fmaf(f.z, f.z, ss);
    ss = fmaf(f.w, f.w, ss);
  };
#pragma unroll
  for (int c = 0; c < kRowCache; ++c) {
    const int i = threadIdx.x + c * blockDim.x;
    if (i < v4) {
      xc[c] = load(i);
      acc_ss(xc[c]);
    }
  }
  for (int i = threadIdx.x + kRowCache * blockDim.x; i < v4; i += blockDim.x) acc_ss(load(i));
  float inv = 1.0f;
  if (a.apply_norm) {
    ss = block_sum(ss, red);
    inv = 1.0f / sqrtf(ss / static_cast<float>(a.d) + a.eps);
  }
  T* out = static_cast<T*>(a.out);
  const size_t oo = static_cast<size_t>(row) * a.ld_out;
  // four consecutive outputs at once: one 8-byte (bf16) or 16-byte store per
  // output tensor where the row stride allows (ld_out % 4 == 0, checked on the
  // host), else one store per element
  auto emit = [&](int i, const float4& f4, const float* g) {
    const float f[4] = {f4.x, f4.y, f4.z, f4.w};
    float y[4], st[4];
    T hi[4];
    bf16 lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      y[k] = a.apply_norm ? f[k] * inv * g[k] : f[k];
      st[k] = y[k];
      if (out) {
        hi[k] = Elem<T>::from_f(y[k]);
        st[k] = Elem<T>::to_f(hi[k]);
        if (a.out_lo) {
          lo[k] = __float2bfloat16_rn(y[k] - st[k]);
          st[k] += __bfloat162float(lo[k]);
        }
      }
    }
    const size_t c0 = oo + 4 * static_cast<size_t>(i);
    if (a.vec4) {
      if (out) {
        if constexpr (sizeof(T) == 2) {
          *reinterpret_cast<uint2*>(out + c0) = make_uint2(pack2(hi[0], hi[1]), pack2(hi[2], hi[3]));
        } else {
          *reinterpret_cast<float4*>(out + c0) = make_float4(hi[0], hi[1], hi[2], hi[3]);
        }
        if (a.out_lo)
          *reinterpret_cast<uint2*>(a.out_lo + c0) = make_uint2(pack2(lo[0], lo[1]), pack2(lo[2], lo[3]));
      }
      if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + c0) = make_float4(st[0], st[1], st[2], st[3]);
      if (a.norm_out) *reinterpret_cast<float4*>(a.norm_out + c0) = make_float4(y[0], y[1], y[2], y[3]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (out) {
          out[c0 + k] = hi[k];
          if (a.out_lo) a.out_lo[c0 + k] = lo[k];
        }
        if (a.out_f32) a.out_f32[c0 + k] = st[k];
        if (a.norm_out) a.norm_out[c0 + k] = y[k];
      }
    }
  };
#pragma unroll
  for (int c = 0; c < kRowCache; ++c) {
    const int i = threadIdx.x + c * blockDim.x;
    if (i < v4) emit(i, xc[c], gc[c]);
  }
  for (int i = threadIdx.x + kRowCache * blockDim.x; i < v4; i += blockDim.x) {
    // rows wider than the register cache: the sum again (sum_out is rewritten
    // with the same value)
    float g[4] = {1.f, 1.f, 1.f, 1.f};
    if (a.apply_norm) load_gain4<T>(gam, i, g);
    emit(i, load(i), g);
  }
}

int launch_rownorm(const RowNormArgs& a_in, int dtype, cudaStream_t st) {
  if (a_in.rows_cap <= 0) return PE_OK;
  RowNormArgs a = a_in;
  // vector stores: every output row starts 16-byte aligned
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  a.vec4 = (a.ld_out % 4 == 0) && (!a.out || al16(a.out)) && (!a.out_lo || al16(a.out_lo)) &&
           (!a.out_f32 || al16(a.out_f32)) && (!a.norm_out || al16(a.norm_out));
  const int threads = a.d >= 2048 ? 256 : 128;
  const cudaError_t e =
      dtype == PE_DTYPE_BF16
          ? launch_pdl(rownorm_kernel<bf16>, dim3(a.rows_cap), dim3(threads), 0, st, a)
          : launch_pdl(rownorm_kernel<float>, dim3(a.rows_cap), dim3(threads), 0, st, a);
  return e == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

// ------------------------------------------------------------------ RoPE + KV write

// CTAs (v, y): non-rejected row v, the y-th of gridDim.y slices of its heads
// (every element sums the QKV partial tiles, so a few rows are spread over
// several CTAs each).  The row is a sample row when it is one of the last K
// non-rejected rows of its request (NTP row + MASK rows).
constexpr int kRopeCtasPerRow = 8;  // at most
// CTAs per row: as many as one wave of 8 CTAs per SM holds for all rows (a row
// has only (H + 2G) hd / 2 rotations: a CTA's fixed chain of dependent loads,
// not its elements, sets its time), at least 1, at most kRopeCtasPerRow
int rope_ctas_per_row(int rows) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return std::max(1, std::min(kRopeCtasPerRow, 8 * std::max(sms, 1) / rows));
}

template <typename T>
__global__ void __launch_bounds__(256) rope_kv_kernel(const RopeArgs a) {
  __shared__ float cs[64], sn[64];
  __shared__ int samp_sh;
  pdl_trigger();
  pdl_wait();
  const int half = a.hd / 2;
  int v;  // the non-rejected row this CTA rotates
  if (a.padded_in) {
    // right-aligned rows: row blockIdx.x = r * K + k of request r
    const int r = blockIdx.x / a.K, k = blockIdx.x - r * a.K;
    v = a.valid_qsl[r + 1] - a.K + k;
    if (v < a.valid_qsl[r]) {
      // padding row: a zero query (its output is never used), no KV
      T* q = static_cast<T*>(a.q_s) + static_cast<size_t>(blockIdx.x) * a.H * a.hd;
      const int tid = blockIdx.y * blockDim.x + threadIdx.x;
      for (int e = tid; e < a.H * a.hd; e += gridDim.y * blockDim.x) q[e] = Elem<T>::from_f(0.f);
      return;
    }
  } else {
    v = blockIdx.x;
    const int nv = min(max(*a.n_valid, 0), a.T_out);
    if (v >= nv) return;
  }
  const int o = a.valid_rows[v];
  if (o < 0 || o >= a.T_out) {
    if (threadIdx.x == 0) set_status(a.status, PE_ST_ACCEPTED_RANGE);
    return;
  }
  const int64_t p = a.pos[o];
  const int64_t slot = a.slot[o];
  if (threadIdx.x < 32) {
    if (a.padded_in) {
      if (threadIdx.x == 0) samp_sh = blockIdx.x;
    } else {
      // request of row v: the requests whose first non-rejected row is at or
      // before v, less one (valid_qsl rises strictly: each request keeps at
      // least K rows).  The warp compares 32 offsets per round with one ballot;
      // the rounds' loads are independent, so a batch costs one or two load
      // latencies instead of a binary search's log2(B) dependent loads.
      const int lane = threadIdx.x;
      int cnt = 0;
#pragma unroll 4
      for (int base = 0; base < a.B; base += 32) {
        const int i = base + lane;
        cnt += __popc(__ballot_sync(0xffffffffu, i < a.B && a.valid_qsl[i] <= v));
      }
      if (lane == 0) {
        const int r = cnt - 1;
        const int k = v - (a.valid_qsl[r + 1] - a.K);
        samp_sh = (k >= 0 && k < a.K) ? r * a.K + k : -1;
        if (k < 0 && a.must_fit && blockIdx.y == 0) set_status(a.status, PE_ST_ROWS_RANGE);
      }
    }
  }
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    float s, c;
    rope_cos_sin(p, a.rope_turn[i], c, s);
    cs[i] = c;
    sn[i] = s;
  }
  __syncthreads();
  const int s_idx = samp_sh;
  const int QKV = (a.H + 2 * a.G) * a.hd;
  const int tid = blockIdx.y * blockDim.x + threadIdx.x;  // thread within the row
  const int nthr = gridDim.y * blockDim.x;
  // element x of this row of the QKV projection: the sum of its partial tiles
  const float* row0 = a.qkv + static_cast<size_t>(a.padded_in ? blockIdx.x : v) * QKV;
  auto qkv_at = [&](int x) {
    float acc = 0.f;
    for (int k = 0; k < a.n_parts; ++k) acc += row0[k * a.part_stride + x];
    return acc;
  };
  const bool slot_ok = slot >= 0 && slot < static_cast<int64_t>(a.num_blocks) * a.bs;
  if (!slot_ok && slot != PE_PADDING_SLOT_ID && threadIdx.x == 0)
    set_status(a.status, PE_ST_BLOCK_RANGE);
  const int64_t blk = slot_ok ? slot / a.bs : 0, off = slot_ok ? slot % a.bs : 0;
  if (a.vec4) {
    // four consecutive elements at once (16-byte partial loads, 8- or 16-byte
    // stores; the host checked the strides and alignments)
    auto qkv_at4 = [&](int x, float* f) {
      float4 acc = *reinterpret_cast<const float4*>(row0 + x);
      for (int k = 1; k < a.n_parts; ++k) {
        const float4 p = *reinterpret_cast<const float4*>(row0 + k * a.part_stride + x);
        acc.x += p.x;
        acc.y += p.y;
        acc.z += p.z;
        acc.w += p.w;
      }
      f[0] = acc.x;
      f[1] = acc.y;
      f[2] = acc.z;
      f[3] = acc.w;
    };
    const int q4 = half / 4;
    for (int e = tid; e < (a.H + a.G) * q4; e += nthr) {
      const int hh = e / q4, i0 = (e - hh * q4) * 4;
      float x1[4], x2[4], y1[4], y2[4];
      qkv_at4(hh * a.hd + i0, x1);
      qkv_at4(hh * a.hd + i0 + half, x2);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        y1[k] = x1[k] * cs[i0 + k] - x2[k] * sn[i0 + k];
        y2[k] = x2[k] * cs[i0 + k] + x1[k] * sn[i0 + k];
      }
      T* dst = nullptr;
      if (hh < a.H) {
        if (s_idx >= 0) dst = static_cast<T*>(a.q_s) + (static_cast<size_t>(s_idx) * a.H + hh) * a.hd;
      } else if (slot_ok) {
        dst = static_cast<T*>(a.k_cache) + ((blk * a.G + (hh - a.H)) * a.bs + off) * a.hd;
      }
      if (dst) {
        store4<T>(dst + i0, y1);
        store4<T>(dst + i0 + half, y2);
      }
    }
    if (slot_ok) {
      const int v4 = a.hd / 4;
      for (int e = tid; e < a.G * v4; e += nthr) {
        const int g = e / v4, i0 = (e - g * v4) * 4;
        float f[4];
        qkv_at4((a.H + a.G) * a.hd + g * a.hd + i0, f);
        store4<T>(static_cast<T*>(a.v_cache) + ((blk * a.G + g) * a.bs + off) * a.hd + i0, f);
      }
    }
  } else {
  // rotated q (sample rows) and k (all rows)
  for (int e = tid; e < (a.H + a.G) * half; e += nthr) {
    const int hh = e / half, i = e - hh * half;
    const float x1 = qkv_at(hh * a.hd + i), x2 = qkv_at(hh * a.hd + i + half);
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
    for (int e = tid; e < a.G * a.hd; e += nthr) {
      const int g = e / a.hd, i = e - g * a.hd;
      T* vc = static_cast<T*>(a.v_cache) + ((blk * a.G + g) * a.bs + off) * a.hd;
      vc[i] = Elem<T>::from_f(qkv_at((a.H + a.G) * a.hd + e));
    }
  }
  }
  if (s_idx >= 0 && a.x_s) {
    // the fc output of the sample rows is the attention residual (fp32)
    const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(v) * a.d);
    float4* dst = reinterpret_cast<float4*>(a.x_s + static_cast<size_t>(s_idx) * a.d);
    for (int i = tid; i < a.d / 4; i += nthr) dst[i] = src[i];
  }
}

int launch_rope_kv(const RopeArgs& a, int dtype, cudaStream_t st) {
  const int rows = a.padded_in ? a.B * a.K : a.T_out;
  if (rows <= 0) return PE_OK;
  const dim3 grid(rows, rope_ctas_per_row(rows));
  RopeArgs av = a;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  const size_t esz = dtype == PE_DTYPE_BF16 ? 2 : 4;
  // 16-byte partial loads need every row and part to start 16-byte aligned;
  // 4-element stores need hd % 8 == 0 (so half % 4 == 0) and aligned rows
  av.vec4 = a.hd % 8 == 0 && (static_cast<size_t>(a.H + 2 * a.G) * a.hd) % 4 == 0 &&
            a.part_stride % 4 == 0 && al16(a.qkv) && al16(a.q_s) && al16(a.k_cache) &&
            al16(a.v_cache) && (static_cast<size_t>(a.hd) * esz) % 8 == 0;
  const cudaError_t e =
      dtype == PE_DTYPE_BF16
          ? launch_pdl(rope_kv_kernel<bf16>, grid, dim3(256), 0, st, av)
          : launch_pdl(rope_kv_kernel<float>, grid, dim3(256), 0, st, av);
  return e == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

// ------------------------------------------------------------------ argmax keys

// A memset node would end the chain of programmatic launches; this kernel keeps
// it, so the LM-head GEMM after it sets up and pulls its first weights into L2
// while the kernels before finish.
__global__ void zero_keys_kernel(unsigned long long* __restrict__ keys, int n) {
  pdl_trigger();
  pdl_wait();  // the previous argmax finalisation may still be reading them
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) keys[i] = 0ull;
}

int launch_zero_keys(unsigned long long* keys, int n, cudaStream_t st) {
  if (n <= 0) return PE_OK;
  const int blocks = std::min((n + 255) / 256, 64);
  return launch_pdl(zero_keys_kernel, dim3(blocks), dim3(256), 0, st, keys, n) == cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}


__global__ void argmax_finalize_kernel(const unsigned long long* __restrict__ keys, int n,
                                       int32_t* __restrict__ out, int stride) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const unsigned long long k = keys[i];
  out[static_cast<size_t>(i) * stride] =
      k ? static_cast<int32_t>(~static_cast<uint32_t>(k & 0xffffffffull)) : 0;
}

int launch_argmax_finalize(const unsigned long long* keys, int n, int32_t* out, cudaStream_t st,
                           int stride) {
  if (n <= 0) return PE_OK;
  return launch_pdl(argmax_finalize_kernel, dim3((n + 255) / 256), dim3(256), 0, st, keys, n, out,
                    stride) == cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}

// ------------------------------------------------------------------ bounded-wait check

// One thread waits, through the bounded mbarrier wait every kernel here uses, on
// a barrier nothing ever arrives on.  The wait gives up after its limit; the
// kernel records PE_ST_TIMEOUT and returns, leaving the context usable.
__global__ void __launch_bounds__(32) bounded_wait_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_sh;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_sh = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, &abort_sh)) set_status(status, PE_ST_TIMEOUT);
}

int launch_bounded_wait(uint32_t* status, cudaStream_t st) {
  bounded_wait_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError() == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

}  // namespace pe
