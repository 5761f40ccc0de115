// Steps (1)-(3) of the parallel-draft step: batch metadata, hidden-state map
// and drafter input ("P-EAGLE: parallel speculative decoding in vLLM": Fused
// Triton kernel, Hidden-state management, KV cache and CUDA graphs;
// "Attention Drift" section 4.1, Observation 2).
//
// Every index read from user data is range-checked: out-of-range values are
// clamped or skipped and reported in the status word, never dereferenced.
#include "pe_common.cuh"
#include "pe_prep.h"

namespace pe {

// ------------------------------------------------------------------ (1) metadata

struct MetaArgs {
  int B, T_in, T_out, K, mask_id, bs, max_blocks, num_blocks, vocab;
  const int32_t* qsl;
  const int32_t* prev_tok;
  const int64_t* prev_pos;
  const int32_t* accepted;
  const int32_t* bonus;
  const int32_t* block_table;
  pe_meta m;
  uint32_t* status;
};

// Per-request row counts, with the input checks (identical in both passes).
PE_DEV void request_counts(const MetaArgs& a, int r, int& n, int& acc, bool& bad) {
  int q0 = a.qsl[r], q1 = a.qsl[r + 1];
  bad = false;
  if (q0 < 0 || q1 > a.T_in || q1 < q0) {
    bad = true;
    q0 = min(max(q0, 0), a.T_in);
    q1 = min(max(q1, q0), a.T_in);
  }
  n = q1 - q0;
  acc = a.accepted[r];
  if (n < 1 || acc < 0 || acc > n - 1) {
    bad = true;
    acc = min(max(acc, 0), max(n - 1, 0));
  }
}

// Cache slot of position p of request r through its block table; -1 (flagged)
// when the position or the block id is out of range.
PE_DEV int64_t slot_of(const MetaArgs& a, int r, int64_t p) {
  if (p < 0 || p / a.bs >= a.max_blocks) {
    set_status(a.status, PE_ST_BLOCK_RANGE);
    return PE_PADDING_SLOT_ID;
  }
  const int blk = a.block_table[static_cast<size_t>(r) * a.max_blocks + p / a.bs];
  if (blk < 0 || blk >= a.num_blocks) {
    set_status(a.status, PE_ST_BLOCK_RANGE);
    return PE_PADDING_SLOT_ID;
  }
  return static_cast<int64_t>(blk) * a.bs + p % a.bs;
}

// Pass 1 (every CTA): exclusive block scans (warp shuffles + one shared-memory
// level) of n_r + K - 1 (output rows) and a_r + K (non-rejected rows) over all
// requests; the requests are few, so each CTA redoes the scan instead of
// waiting for another CTA.  Pass 2: CTA c writes the rows of requests
// [c*R, (c+1)*R), one warp per request (R = warps per CTA).
__global__ void __launch_bounds__(256) meta_kernel(const MetaArgs a) {
  __shared__ int wsum_o[32], wsum_v[32];
  __shared__ int carry_o, carry_v;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = blockDim.x >> 5;
  const int r_begin = blockIdx.x * nw, r_end = min(a.B, r_begin + nw);
  // the batch's inputs may come from the kernel before (the verification):
  // wait for it, and only then let the next kernel start, so that it may read
  // the same inputs without waiting for this kernel
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    carry_o = 0;
    carry_v = 0;
  }
  __syncthreads();
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int r = base + tid;
    int lo = 0, lv = 0;
    if (r < a.B) {
      int n, acc;
      bool bad;
      request_counts(a, r, n, acc, bad);
      if (bad && r >= r_begin && r < r_end) set_status(a.status, PE_ST_ACCEPTED_RANGE);
      lo = n + a.K - 1;
      lv = (n >= 1 ? acc + 1 : 0) + a.K - 1;
    }
    int xo = lo, xv = lv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int to = __shfl_up_sync(0xffffffffu, xo, off);
      const int tv = __shfl_up_sync(0xffffffffu, xv, off);
      if (lane >= off) {
        xo += to;
        xv += tv;
      }
    }
    if (lane == 31) {
      wsum_o[warp] = xo;
      wsum_v[warp] = xv;
    }
    __syncthreads();
    if (warp == 0) {
      int so = lane < nw ? wsum_o[lane] : 0;
      int sv = lane < nw ? wsum_v[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int to = __shfl_up_sync(0xffffffffu, so, off);
        const int tv = __shfl_up_sync(0xffffffffu, sv, off);
        if (lane >= off) {
          so += to;
          sv += tv;
        }
      }
      if (lane < nw) {
        wsum_o[lane] = so;  // inclusive prefix of warp totals
        wsum_v[lane] = sv;
      }
    }
    __syncthreads();
    const int pre_o = carry_o + (warp ? wsum_o[warp - 1] : 0) + xo - lo;
    const int pre_v = carry_v + (warp ? wsum_v[warp - 1] : 0) + xv - lv;
    if (r < a.B && (r >= r_begin && r < r_end)) {
      a.m.out_qsl[r] = pre_o;
      a.m.valid_qsl[r] = pre_v;
    }
    __syncthreads();
    if (tid == 0) {
      carry_o += wsum_o[nw - 1];
      carry_v += wsum_v[nw - 1];
    }
    __syncthreads();
  }
  if (tid == 0 && blockIdx.x == 0) {
    a.m.out_qsl[a.B] = carry_o;
    a.m.valid_qsl[a.B] = carry_v;
    *a.m.n_valid = min(carry_v, a.T_out);
    if (carry_o != a.T_out) set_status(a.status, PE_ST_ACCEPTED_RANGE);
  }
  __syncthreads();

  // pass 2: rows of request r (this CTA's own requests; their offsets were
  // written by this CTA above)
  for (int r = r_begin + warp; r < r_end; r += nw) {
    int n, acc;
    bool bad;
    request_counts(a, r, n, acc, bad);
    const int q0 = min(max(a.qsl[r], 0), a.T_in);
    const int o0 = a.m.out_qsl[r];
    const int v0 = a.m.valid_qsl[r];
    const int b = a.bonus[r];
    if (b < 0 || b >= a.vocab) set_status(a.status, PE_ST_TOKEN_RANGE);
    const int i_ntp = min(q0 + acc, a.T_in - 1);
    const int64_t p0 = a.prev_pos[i_ntp];
    const int rows = n + a.K - 1;
    for (int j = lane; j < rows; j += 32) {
      const int o = o0 + j;
      if (o < 0 || o >= a.T_out) {
        set_status(a.status, PE_ST_ACCEPTED_RANGE);
        continue;
      }
      int tok, hsrc, vi = -1;
      int64_t pos, slot;
      uint8_t rej = 0, msk = 0;
      if (j < n) {
        const int i = q0 + j;
        tok = (j == acc || j == n - 1) ? b : a.prev_tok[i + 1];
        if (j != acc && j != n - 1 && (tok < 0 || tok >= a.vocab))
          set_status(a.status, PE_ST_TOKEN_RANGE);
        pos = a.prev_pos[i];
        hsrc = i;
        if (j > acc) {
          rej = 1;
          slot = PE_PADDING_SLOT_ID;
        } else {
          slot = slot_of(a, r, pos);
          vi = v0 + j;
        }
        if (j == acc) a.m.sample_idx[static_cast<size_t>(r) * a.K] = o;
      } else {
        const int mm = j - n + 1;  // 1..K-1
        tok = a.mask_id;
        pos = p0 + mm;
        hsrc = -1;
        msk = 1;
        slot = slot_of(a, r, pos);
        vi = v0 + acc + mm;
        a.m.sample_idx[static_cast<size_t>(r) * a.K + mm] = o;
      }
      a.m.tok[o] = tok;
      a.m.pos[o] = pos;
      a.m.is_rejected[o] = rej;
      a.m.is_masked[o] = msk;
      a.m.hidden_src[o] = hsrc;
      a.m.slot[o] = slot;
      if (vi >= 0) {
        if (vi < a.T_out)
          a.m.valid_rows[vi] = o;
        else
          set_status(a.status, PE_ST_ACCEPTED_RANGE);
      }
    }
    if (lane == 0) a.m.seq_len[r] = static_cast<int32_t>(p0 + a.K);
  }
  // rows past the non-rejected count (every CTA knows the total)
  const int nv = min(carry_v, a.T_out);
  for (int i = nv + blockIdx.x * blockDim.x + tid; i < a.T_out; i += gridDim.x * blockDim.x)
    a.m.valid_rows[i] = -1;
}

int launch_meta(const MetaLaunch& L, cudaStream_t st) {
  MetaArgs a;
  a.B = L.B;
  a.T_in = L.T_in;
  a.T_out = L.T_in + L.B * (L.K - 1);
  a.K = L.K;
  a.mask_id = L.mask_id;
  a.bs = L.bs;
  a.max_blocks = L.max_blocks;
  a.num_blocks = L.num_blocks;
  a.vocab = L.vocab;
  a.qsl = L.qsl;
  a.prev_tok = L.prev_tok;
  a.prev_pos = L.prev_pos;
  a.accepted = L.accepted;
  a.bonus = L.bonus;
  a.block_table = L.block_table;
  a.m = L.meta;
  a.status = L.status;
  // 8 warps per CTA, one request per warp in pass 2
  const int threads = 256;
  const int grid = (L.B + threads / 32 - 1) / (threads / 32);
  return launch_pdl(meta_kernel, dim3(grid), dim3(threads), 0, st, a) == cudaSuccess ? PE_OK
                                                                                  : PE_ERR_CUDA;
}

// ------------------------------------------------------------------ (2) hidden-state map

// G[o][s][:] = H_tgt[hidden_src[o]][s][:] or h_shared; E[o][:] = emb[tok[o]] or
// emb_mask.  Grid-stride over 16-byte vectors; 4 loads in flight per thread.
template <typename T>
__global__ void __launch_bounds__(256) gather_kernel(GatherArgs a) {
  pdl_trigger();
  pdl_wait();
  constexpr int V = Elem<T>::kVec;
  const int vd = a.d / V;             // vectors per stream row
  const long nG = a.G ? static_cast<long>(a.T_out) * 3 * vd : 0;
  const long nE = a.E ? static_cast<long>(a.T_out) * vd : 0;
  const long total = nG + nE;
  const long stride = static_cast<long>(gridDim.x) * blockDim.x;
  const uint4* H = static_cast<const uint4*>(a.H_tgt);
  const uint4* hs = static_cast<const uint4*>(a.h_shared);
  const uint4* emb = static_cast<const uint4*>(a.emb);
  const uint4* em = static_cast<const uint4*>(a.emb_mask);
  for (long base = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; base < total;
       base += 4 * stride) {
    uint4 val[4];
    long dst[4];
    bool isG[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long idx = base + u * stride;
      dst[u] = -1;
      if (idx >= total) continue;
      if (idx < nG) {
        const long o = idx / (3 * vd);
        const int rem = static_cast<int>(idx - o * 3 * vd);
        const int src = a.hidden_src[o];
        if (src >= 0 && src < a.T_in)
          val[u] = H[static_cast<long>(src) * 3 * vd + rem];
        else if (src < 0)
          val[u] = hs[rem % vd];
        else {
          set_status(a.status, PE_ST_ACCEPTED_RANGE);
          val[u] = make_uint4(0, 0, 0, 0);
        }
        dst[u] = idx;
        isG[u] = true;
      } else {
        const long e = idx - nG;
        const long o = e / vd;
        const int rem = static_cast<int>(e - o * vd);
        if (a.is_masked[o]) {
          val[u] = em[rem];
        } else {
          int t = a.tok[o];
          if (t < 0 || t >= a.vocab) {
            set_status(a.status, PE_ST_TOKEN_RANGE);
            t = 0;
          }
          val[u] = emb[static_cast<long>(t) * vd + rem];
        }
        dst[u] = e;
        isG[u] = false;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (dst[u] < 0) continue;
      if (isG[u])
        static_cast<uint4*>(a.G)[dst[u]] = val[u];
      else
        static_cast<uint4*>(a.E)[dst[u]] = val[u];
    }
  }
}

// ------------------------------------------------------------------ (3) drafter input

// A[v] = [RMSNorm(G0) g0, RMSNorm(G1) g1, RMSNorm(G2) g2, E] for non-rejected row
// v (output row valid_rows[v]), straight from H_tgt / h_shared / the embedding.
// One CTA of 8 warps per row: warps 2s and 2s+1 write segment s (0..2 the
// streams, 3 the embedding), so a row's four segments load together and a
// wave of CTAs covers hundreds of rows.  Each thread keeps up to kInputVecs
// vectors of its segment in registers (segments of up to 8 * 64 * 8 = 4096 bf16
// elements; longer ones read the rest twice).
constexpr int kInputVecs = 8;
constexpr int kInputThreads = 256;
constexpr int kSegThreads = 64;

// Warp 0 of an input CTA: the request, hidden source and token of non-rejected
// row v, from the verify batch itself.  The per-request counts take the metadata
// kernel's clamps (request_counts), so row v is the one that kernel lists at
// valid_rows[v]: request r's copied rows 0..a_r, then its K-1 MASK rows.
// out[0] = 1 when v exists; out[1] = hidden source (-1: h_shared), out[2] =
// token, out[3] = 1 for a MASK row.
PE_DEV void locate_valid_row(const InputArgs& a, int v, int* out) {
  const int lane = threadIdx.x & 31;
  int base = 0, found = 0, hsrc = -1, tok = 0, masked = 1;
  for (int r0 = 0; r0 < a.B; r0 += 32) {
    const int r = r0 + lane;
    int q0 = 0, n = 0, acc = 0, c = 0;
    if (r < a.B) {
      q0 = a.qsl[r];
      int q1 = a.qsl[r + 1];
      if (q0 < 0 || q1 > a.T_in || q1 < q0) {
        q0 = min(max(q0, 0), a.T_in);
        q1 = min(max(q1, q0), a.T_in);
      }
      n = q1 - q0;
      acc = a.accepted[r];
      if (n < 1 || acc < 0 || acc > n - 1) acc = min(max(acc, 0), max(n - 1, 0));
      c = (n >= 1 ? acc + 1 : 0) + a.K - 1;
    }
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    const int start = base + incl - c;
    const bool hit = r < a.B && v >= start && v < start + c;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (hit) {
      const int j = v - start;
      if (n >= 1 && j <= acc) {
        hsrc = q0 + j;
        tok = (j == acc || j == n - 1) ? a.bonus[r] : a.prev_tok[q0 + j + 1];
        masked = 0;
      }
    }
    if (m) {
      const int src = __ffs(static_cast<int>(m)) - 1;
      hsrc = __shfl_sync(0xffffffffu, hsrc, src);
      tok = __shfl_sync(0xffffffffu, tok, src);
      masked = __shfl_sync(0xffffffffu, masked, src);
      found = 1;
      break;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    out[0] = found && v < a.T_out;
    out[1] = hsrc;
    out[2] = tok;
    out[3] = masked;
  }
}

template <typename T>
__global__ void __launch_bounds__(kInputThreads) input_kernel(InputArgs a) {
  __shared__ float red[4][2];
  __shared__ int row_sh[4];
  constexpr int V = Elem<T>::kVec;
  const int v = blockIdx.x;
  const int vd = a.d / V;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = warp >> 1;
  const int st = tid & (kSegThreads - 1);  // thread within the segment
  // the gains are weights, independent of the kernels before: read them first
  uint4 g[kInputVecs];
  const uint4* gam = static_cast<const uint4*>(a.gamma_stream) + static_cast<size_t>(seg) * vd;
  if (seg < 3) {
#pragma unroll
    for (int c = 0; c < kInputVecs; ++c) {
      const int i = st + c * kSegThreads;
      if (i < vd) g[c] = gam[i];
    }
  }
  pdl_trigger();
  if (a.self_index) {
    // the metadata kernel let this kernel start after its own dependency wait:
    // the verify batch is final, and its outputs are not needed
    if (warp == 0) locate_valid_row(a, v, row_sh);
  } else if (tid == 0) {
    pdl_wait();
    const int nv = min(max(*a.n_valid, 0), a.T_out);
    int ok = v < nv;
    int o = ok ? a.valid_rows[v] : -1;
    if (ok && (o < 0 || o >= a.T_out)) {
      set_status(a.status, PE_ST_ACCEPTED_RANGE);
      ok = 0;
    }
    row_sh[0] = ok;
    if (ok) {
      row_sh[1] = a.hidden_src[o];
      row_sh[2] = a.tok[o];
      row_sh[3] = a.is_masked[o];
    }
  }
  __syncthreads();
  if (!row_sh[0]) {
    if (a.self_index) pdl_wait();
    return;
  }
  const int hsrc = row_sh[1], tok = row_sh[2], masked = row_sh[3];
  uint4* out = reinterpret_cast<uint4*>(static_cast<T*>(a.A) + static_cast<size_t>(v) * 4 * a.d +
                                        static_cast<size_t>(seg) * a.d);
  const uint4* src;
  if (seg == 3) {
    if (masked) {
      src = static_cast<const uint4*>(a.emb_mask);
    } else {
      int t = tok;
      if (t < 0 || t >= a.vocab) {
        if (st == 0) set_status(a.status, PE_ST_TOKEN_RANGE);
        t = 0;
      }
      src = static_cast<const uint4*>(a.emb) + static_cast<size_t>(t) * vd;
    }
  } else if (hsrc < 0) {
    src = static_cast<const uint4*>(a.h_shared);
  } else if (hsrc < a.T_in) {
    src = static_cast<const uint4*>(a.H_tgt) + (static_cast<size_t>(hsrc) * 3 + seg) * vd;
  } else {
    if (st == 0) set_status(a.status, PE_ST_ACCEPTED_RANGE);
    src = static_cast<const uint4*>(a.h_shared);
  }
  // the segment's vectors i = st, st + 64, ...: the first kInputVecs stay in
  // registers (all loads in flight together), summed in that order
  uint4 x[kInputVecs];
#pragma unroll
  for (int c = 0; c < kInputVecs; ++c) {
    const int i = st + c * kSegThreads;
    if (i < vd) x[c] = src[i];
  }
  float ss = 0.f;
  if (seg < 3) {
#pragma unroll
    for (int c = 0; c < kInputVecs; ++c) {
      if (st + c * kSegThreads < vd) {
        float f[V];
        unpack16<T>(x[c], f);
#pragma unroll
        for (int k = 0; k < V; ++k) ss = fmaf(f[k], f[k], ss);
      }
    }
    for (int i = st + kInputVecs * kSegThreads; i < vd; i += kSegThreads) {
      float f[V];
      unpack16<T>(src[i], f);
#pragma unroll
      for (int k = 0; k < V; ++k) ss = fmaf(f[k], f[k], ss);
    }
  }
  // the segment's sum of squares: its two warps, then across them
  ss = warp_sum(ss);
  if (lane == 0) red[seg][warp & 1] = ss;
  __syncthreads();
  if (seg == 3) {
    // the embedding row (or emb(mask)) is copied as it is
#pragma unroll
    for (int c = 0; c < kInputVecs; ++c) {
      const int i = st + c * kSegThreads;
      if (i < vd) out[i] = x[c];
    }
    for (int i = st + kInputVecs * kSegThreads; i < vd; i += kSegThreads) out[i] = src[i];
  } else {
    const float inv = 1.0f / sqrtf((red[seg][0] + red[seg][1]) / static_cast<float>(a.d) + a.eps);
#pragma unroll
    for (int c = 0; c < kInputVecs; ++c) {
      const int i = st + c * kSegThreads;
      if (i < vd) {
        float f[V], gf[V];
        unpack16<T>(x[c], f);
        unpack16<T>(g[c], gf);
#pragma unroll
        for (int k = 0; k < V; ++k) f[k] = f[k] * inv * gf[k];
        out[i] = pack16<T>(f);
      }
    }
    for (int i = st + kInputVecs * kSegThreads; i < vd; i += kSegThreads) {
      float f[V], gf[V];
      unpack16<T>(src[i], f);
      unpack16<T>(gam[i], gf);
#pragma unroll
      for (int k = 0; k < V; ++k) f[k] = f[k] * inv * gf[k];
      out[i] = pack16<T>(f);
    }
  }
  // (self-indexed) this kernel completes only after the metadata kernel, so
  // the kernels after it see both
  if (a.self_index) pdl_wait();
}

template <typename T>
int launch_gather_t(const GatherArgs& a, int num_sms, cudaStream_t st) {
  const int vd = a.d / Elem<T>::kVec;
  const long total = static_cast<long>(a.T_out) * vd * ((a.G ? 3 : 0) + (a.E ? 1 : 0));
  if (total == 0) return PE_OK;
  long blocks = (total + 4L * 256 - 1) / (4L * 256);
  blocks = blocks < 4L * num_sms ? blocks : 4L * num_sms;
  return launch_pdl(gather_kernel<T>, dim3(static_cast<int>(blocks)), dim3(256), 0, st, a) ==
                 cudaSuccess
             ? PE_OK
             : PE_ERR_CUDA;
}

int launch_gather(const GatherArgs& a, int dtype, int num_sms, cudaStream_t st) {
  return dtype == PE_DTYPE_BF16 ? launch_gather_t<bf16>(a, num_sms, st)
                                : launch_gather_t<float>(a, num_sms, st);
}

// ------------------------------------------------------------------ autoregressive pass input
// Grid (B, 4): CTA (r, s) writes segment s of request r's row; CTA (r, 0) also
// writes the row's metadata.  The three stream segments normalise the same fp32
// hidden state (each with its own gain), as the parallel step does with
// h_shared in a MASK row.
template <typename T>
__global__ void __launch_bounds__(128) ar_input_kernel(ArInputArgs a) {
  __shared__ float red[32];
  constexpr int V = Elem<T>::kVec;
  const int r = blockIdx.x, seg = blockIdx.y;
  const int vd = a.d / V;
  const int tid = threadIdx.x;
  pdl_trigger();
  pdl_wait();
  int t = a.drafts[static_cast<size_t>(r) * a.K + (a.k - 2)];
  const bool t_ok = t >= 0 && t < a.vocab;
  if (!t_ok) t = 0;
  if (seg == 0 && tid == 0) {
    pe_meta& m = a.meta;
    const int64_t p = a.pos1[a.sample1[r]] + (a.k - 1);
    int64_t slot = PE_PADDING_SLOT_ID;
    const int64_t bi = p >= 0 ? p / a.bs : -1;
    if (bi >= 0 && bi < a.max_blocks) {
      const int blk = a.block_table[static_cast<size_t>(r) * a.max_blocks + bi];
      if (blk >= 0 && blk < a.num_blocks) slot = static_cast<int64_t>(blk) * a.bs + p % a.bs;
    }
    if (slot < 0) set_status(a.status, PE_ST_BLOCK_RANGE);
    if (!t_ok) set_status(a.status, PE_ST_TOKEN_RANGE);
    m.tok[r] = t;
    m.pos[r] = p;
    m.slot[r] = slot;
    m.is_rejected[r] = 0;
    m.is_masked[r] = 0;
    m.hidden_src[r] = -1;
    m.valid_rows[r] = r;
    m.sample_idx[r] = r;
    m.seq_len[r] = static_cast<int32_t>(p + 1);
    m.out_qsl[r] = r;
    m.valid_qsl[r] = r;
    if (r == a.B - 1) {
      m.out_qsl[a.B] = a.B;
      m.valid_qsl[a.B] = a.B;
      *m.n_valid = a.B;
    }
  }
  uint4* out = reinterpret_cast<uint4*>(static_cast<T*>(a.A) + static_cast<size_t>(r) * 4 * a.d +
                                        static_cast<size_t>(seg) * a.d);
  if (seg == 3) {
    const uint4* src = static_cast<const uint4*>(a.emb) + static_cast<size_t>(t) * vd;
    for (int i = tid; i < vd; i += blockDim.x) out[i] = src[i];
    return;
  }
  const float* h = a.hidden + static_cast<size_t>(r) * a.d;
  float ss = 0.f;
  for (int i = tid; i < a.d / 4; i += blockDim.x) {
    const float4 f = reinterpret_cast<const float4*>(h)[i];
    ss = fmaf(f.x, f.x, ss);
    ss = fmaf(f.y, f.y, ss);
    ss = fmaf(f.z, f.z, ss);
    ss = fmaf(f.w, f.w, ss);
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(a.d) + a.eps);
  const uint4* gam = static_cast<const uint4*>(a.gamma_stream) + static_cast<size_t>(seg) * vd;
  for (int i = tid; i < vd; i += blockDim.x) {
    float f[V], gf[V];
#pragma unroll
    for (int k = 0; k < V; ++k) f[k] = h[i * V + k];
    unpack16<T>(gam[i], gf);
#pragma unroll
    for (int k = 0; k < V; ++k) f[k] = f[k] * inv * gf[k];
    out[i] = pack16<T>(f);
  }
}

int launch_ar_input(const ArInputArgs& a, int dtype, cudaStream_t st) {
  if (a.B <= 0) return PE_OK;
  dim3 grid(a.B, 4);
  const cudaError_t e = dtype == PE_DTYPE_BF16
                            ? launch_pdl(ar_input_kernel<bf16>, grid, dim3(128), 0, st, a)
                            : launch_pdl(ar_input_kernel<float>, grid, dim3(128), 0, st, a);
  return e == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

int launch_input(const InputArgs& a, int dtype, cudaStream_t st) {
  if (a.T_out <= 0) return PE_OK;
  dim3 grid(a.T_out);
  const cudaError_t e = dtype == PE_DTYPE_BF16
                            ? launch_pdl(input_kernel<bf16>, grid, dim3(kInputThreads), 0, st, a)
                            : launch_pdl(input_kernel<float>, grid, dim3(kInputThreads), 0, st, a);
  return e == cudaSuccess ? PE_OK : PE_ERR_CUDA;
}

}  // namespace pe
