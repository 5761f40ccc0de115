// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pe.h"

#if __has_include(<nvtx3/nvToolsExt.h>)
#include <nvtx3/nvToolsExt.h>
#define PE_HAVE_NVTX 1
#endif

namespace pe {

// An NVTX range over the enqueue of one C-ABI call, so that a profiler can pick
// out a call's kernels (ncu --nvtx --nvtx-include "pe_argmax/").  Without a tool
// attached the push and pop do nothing.
struct NvtxRange {
  explicit NvtxRange(const char* name) {
#ifdef PE_HAVE_NVTX
    nvtxRangePushA(name);
#else
    (void)name;
#endif
  }
  ~NvtxRange() {
#ifdef PE_HAVE_NVTX
    nvtxRangePop();
#endif
  }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ------------------------------------------------------------------ GEMM epilogues
// Every drafter projection is D[t][f] = sum_k X[t][k] * W[f][k] (X: token rows,
// W: [out][in] weight rows); the epilogue decides what is stored.
enum EpiMode {
  EPI_STORE = 0,        // out[t][f] = D                      (element type of the step)
  EPI_STORE_F32 = 1,    // out[t][f] = D                      (float)
  EPI_RESID_F32 = 2,    // out[t][f] = D + resid[t][f]        (float, float residual)
  EPI_SWIGLU = 3,       // out[t][f] = silu(D_gate) * D_up    (element type of the step)
  EPI_SWIGLU_PAIR = 4,  // the same product as a bf16 pair: out = hi, out2 = lo
  EPI_ARGMAX = 5,       // amax[t] = max over f of key(D, f); optional fp32 logits
  // split k of a K-split GEMM stores its partial sum: out[k * part_stride +
  // t * ld_out + f] (float); the consumer adds the splits in order 0, 1, ...
  EPI_PARTIAL_F32 = 6,
};

struct Epilogue {
  int mode = EPI_STORE;
  void* out = nullptr;
  void* out2 = nullptr;
  int ld_out = 0;
  const float* resid = nullptr;
  int ld_resid = 0;
  unsigned long long* amax = nullptr;
  float* logits = nullptr;
  int ld_logits = 0;
  size_t part_stride = 0;  // EPI_PARTIAL_F32: floats between splits' partial tiles
};

// ------------------------------------------------------------------ tcgen05 GEMM (bf16)
struct TcPlan {
  int M, K, N_cap, dual, bpair;
  int BN, n_tiles, m_tiles, num_kb, k_splits, kb_per_split, stages, grid, tmem_cols;
  int atoms;  // 64-element K atoms per stage
  int acc_bufs;  // TMEM accumulator buffers (2 = the next tile's MMA overlaps the epilogue)
  int ctas_per_sm;  // resident CTAs per SM the plan is sized for
  int partial;      // K splits store partial sums (else they reduce in a cluster)
  int vec;          // wide tiles: the instance whose stores go 4 features at a time
  size_t smem_bytes;
  // unsplit plans with several rounds of tiles: the first main_tiles run
  // persistent, the rest as clusters of tail_splits CTAs splitting K
  int main_tiles, tail_splits, tail_kb_per_split;
};

// partial: the epilogue is EPI_PARTIAL_F32, so splits of K need no cluster (each
// stores its own partial) and the split count is free of cluster limits.
// dual: two weight matrices (gate and up) with two accumulators.  bpair: the
// token rows come as a bf16 pair (hi, lo) whose products add into one accumulator.
TcPlan plan_gemm_tc(int M, int K, int N_cap, int dual, int bpair, int num_sms, bool allow_split,
                    bool partial = false);

// mapA / mapA2: weight tensor maps (box 64 x 128, 128-byte swizzle).  X: token
// rows [N_cap][K] bf16 (row stride K).  n_rows_dev: live token rows on device
// (nullable: all N_cap).  A split plan launches clusters of k_splits CTAs and
// needs no global scratch.
int launch_gemm_tc(const TcPlan& plan, const CUtensorMap* mapA, const CUtensorMap* mapA2,
                   const void* X, const void* X_lo, const int* n_rows_dev, const Epilogue& epi,
                   uint32_t* status, cudaStream_t st);

// ------------------------------------------------------------------ fp32 SIMT GEMM
int launch_gemm_f32(const float* W, const float* W2, const float* X, int M, int K, int N_cap,
                    const int* n_rows_dev, const Epilogue& epi, cudaStream_t st);

// ------------------------------------------------------------------ tensor maps
// Row-major bf16 matrix [rows][cols] -> 2-D tensor map with a box of
// box_rows x 64 elements and the 128-byte swizzle.  Returns false on failure.
bool encode_tmap_bf16(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows);

// ------------------------------------------------------------------ tile-packed weights
// A weight W [M][K] (bf16, row-major) copied into the order the GEMM reads it:
// tile (m, a) = rows 128m..128m+127 x columns 64a..64a+63 is one contiguous
// 16 KB block of 128 rows of 128 bytes; blocks run over a (K) within m.  Rows
// past M and columns past K are zero.  Each weight box the GEMM loads is then
// one contiguous stretch of DRAM rather than 128 stretches of 128 bytes spread
// over the matrix (the weights of a narrow step are streamed once, at DRAM speed).
size_t packed_weight_bytes(int M, int K);
int pack_weight(const void* W, int M, int K, void* P, cudaStream_t st);
// tensor map over a packed weight: [m_tiles * k_atoms * 128 rows][64], box 128 x 64
bool encode_packed_weight_map(CUtensorMap* map, const void* P, int M, int K);

// ------------------------------------------------------------------ persistent decode layer
// A one-layer bf16 step whose token rows (T_out, and B*K sample rows) fit in
// one 16-row tile runs its layer as two persistent kernels around attention
// (pe_decode.cu).
constexpr int kDecodeRows = 16;

struct DecodeLaunch {
  int d, H, G, hd, inter, K, B, T_out, bs, num_blocks, post_norm, num_sms;
  float eps;
  uint64_t rope_turn[64];
  const CUtensorMap* m_fc;
  const CUtensorMap* m_qkv;
  const CUtensorMap* m_o;
  const CUtensorMap* m_gate;
  const CUtensorMap* m_up;
  const CUtensorMap* m_down;
  const void* A;           // part 1 token rows [T_out][4d]
  const int* n_valid;
  const int32_t* valid_rows;
  const int32_t* valid_qsl;
  const int64_t* pos;
  const int64_t* slot;
  const void* gamma_in;
  const void* gamma_post;
  const void* gamma_final;
  void* q_s;               // [B*K][H][hd]
  void* k_cache;
  void* v_cache;
  float* x_s;              // [B*K][d]
  const void* attn;        // part 2 token rows [B*K][H*hd]
  void* z;                 // [B*K][d]
  float* hidden_out;       // nullable
  void* scratch;           // decode_scratch_bytes
  uint32_t* bar;           // 16 barrier words, zero on first use
  uint32_t* status;
};
size_t decode_scratch_bytes(int d, int qkv, int inter, int num_sms);
// whether the decode layer handles these dimensions on this device
bool decode_layer_fits(int d, int qkv, int inter, int num_sms);
// part 1: fc, QKV, RoPE + KV write; part 2: O, gate/up, down, final norm
int launch_decode_layer(const DecodeLaunch& L, int part, cudaStream_t st);

int num_sms_of_current_device();

// Read-only views of a handle (defined beside the handle).
const pe_dims* handle_dims(const pe_handle* h);
const CUtensorMap* handle_lm_map(const pe_handle* h);
int handle_num_sms(const pe_handle* h);
const void* handle_w_lm(const pe_handle* h);
bool handle_has_layer(const pe_handle* h);

}  // namespace pe
