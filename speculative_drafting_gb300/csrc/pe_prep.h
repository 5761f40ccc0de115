// Launch interfaces of the non-GEMM kernels (host side).
#pragma once

#include <cuda_bf16.h>

#include "pe_internal.h"

namespace pe {

typedef __nv_bfloat16 bf16_t;

// ---------------------------------------------------------------- (1) metadata
struct MetaLaunch {
  int B, T_in, K, mask_id, bs, max_blocks, num_blocks, vocab;
  const int32_t* qsl;
  const int32_t* prev_tok;
  const int64_t* prev_pos;
  const int32_t* accepted;
  const int32_t* bonus;
  const int32_t* block_table;
  pe_meta meta;
  uint32_t* status;
};
int launch_meta(const MetaLaunch& L, cudaStream_t st);
// Largest batch for which the drafter-input kernel indexes its rows itself.
constexpr int kSelfIndexMaxBatch = 256;

// ---------------------------------------------------------------- (2) hidden-state map
struct GatherArgs {
  int T_out, T_in, d, vocab;
  const int32_t* hidden_src;
  const int32_t* tok;
  const uint8_t* is_masked;
  const void* H_tgt;
  const void* h_shared;
  const void* emb;
  const void* emb_mask;
  void* G;  // nullable
  void* E;  // nullable
  uint32_t* status;
};
int launch_gather(const GatherArgs& a, int dtype, int num_sms, cudaStream_t st);

// ---------------------------------------------------------------- (3) drafter input
struct InputArgs {
  int T_out, T_in, d, vocab;
  float eps;
  // self_index: each CTA finds its row's request, hidden source and token from
  // the verify batch itself (B, K, qsl, prev_tok, accepted, bonus), with the
  // same clamps as the metadata kernel, instead of waiting for that kernel's
  // outputs; the two kernels then run side by side.  Small batches only (every
  // CTA scans all B requests).
  int self_index, B, K;
  const int32_t* qsl;
  const int32_t* prev_tok;
  const int32_t* accepted;
  const int32_t* bonus;
  const int32_t* n_valid;
  const int32_t* valid_rows;
  const int32_t* hidden_src;
  const int32_t* tok;
  const uint8_t* is_masked;
  const void* H_tgt;
  const void* h_shared;
  const void* emb;
  const void* emb_mask;
  const void* gamma_stream;
  void* A;
  uint32_t* status;
};
int launch_input(const InputArgs& a, int dtype, cudaStream_t st);

// ---------------------------------------------------------------- autoregressive pass input
// Pass k >= 2 of the autoregressive K-pass drafting: one row per request at
// position pos0[r] + k - 1, where pos0[r] = pos1[sample1[r]] is the NTP row's
// position of pass 1.  Its drafter input is [RMSNorm(h)*g0, RMSNorm(h)*g1,
// RMSNorm(h)*g2, emb(t)] with h = hidden[r] (the drafter's own hidden state of
// the previous pass, fp32) and t = drafts[r * K + k - 2]; its metadata (one
// non-rejected row per request, which is also its sample row) goes into meta.
struct ArInputArgs {
  int B, K, k, d, vocab, bs, max_blocks, num_blocks;
  float eps;
  const int64_t* pos1;       // pass 1's row positions
  const int32_t* sample1;    // pass 1's sample row of each request (the NTP row)
  const int32_t* drafts;     // [B][K] draft tokens of the passes so far
  const float* hidden;       // [B][d]
  const int32_t* block_table;
  const void* emb;
  const void* gamma_stream;
  pe_meta meta;              // out: B rows (tok, pos, slot, valid_qsl, valid_rows,
                             // n_valid, sample_idx, seq_len, out_qsl, flags)
  void* A;                   // out: [B][4d]
  uint32_t* status;
};
int launch_ar_input(const ArInputArgs& a, int dtype, cudaStream_t st);

// ---------------------------------------------------------------- row RMSNorm
// y[i] = x[i] * gamma / sqrt(mean(x[i]^2) + eps) (apply_norm) or x[i], for rows
// i < n_rows, where x = (sum of n_parts partial tiles, in order) + resid, stored
// as: out (step dtype), out_lo (bf16 rest of a pair, nullable), out_f32 (fp32
// value of what was stored, nullable); sum_out (nullable) receives x itself.
struct RowNormArgs {
  const float* x;  // partial k of row i at x[k * part_stride + i * ld_x]
  int ld_x;
  int n_parts;
  size_t part_stride;
  const float* resid;  // nullable, [rows][ld_resid]
  int ld_resid;
  float* sum_out;  // nullable, [rows][ld_x]
  float* norm_out; // nullable, [rows][ld_out]: the normalised value before rounding
  const void* gamma;
  int apply_norm;
  void* out;
  bf16_t* out_lo;
  float* out_f32;
  int ld_out, d;
  float eps;
  int rows_cap;
  const int* n_rows_dev;
  // in_group > 0: output row i reads input row (i / out_group) * in_group +
  // (in_group - out_group) + i % out_group, i.e. the last out_group of each
  // group of in_group input rows (the sample rows of a right-aligned layout)
  int in_group, out_group;
  int vec4;  // set by launch_rownorm: four outputs per store
};
int launch_rownorm(const RowNormArgs& a, int dtype, cudaStream_t st);

// ---------------------------------------------------------------- RoPE + KV write
struct RopeArgs {
  int T_out, B, K, H, G, hd, d, bs, num_blocks;
  const float* qkv;  // n_parts partial tiles of [T_out][(H+2G)hd] fp32, part_stride
                     // apart; non-rejected rows in valid_rows order
  int n_parts;
  size_t part_stride;
  const float* x;    // [T_out][d] fc output, fp32 (same order)
  const int32_t* n_valid;
  const int32_t* valid_rows;
  const int32_t* valid_qsl;
  const int64_t* pos;
  const int64_t* slot;
  void* k_cache;
  void* v_cache;
  void* q_s;    // [B*K][H][hd] queries of the sample rows
  float* x_s;  // [B*K][d] fc output of the sample rows (residual, fp32); nullable
  uint64_t rope_turn[64];  // fractions of a turn per position (rope_cos_sin)
  // 0: qkv rows are the non-rejected rows in valid_rows order (K is then the
  // number of rows per request that q_s / x_s keep, right-aligned);
  // 1: qkv rows are already in that right-aligned layout, B*K rows (rows of a
  // request before its first non-rejected row are padding: q = 0, no KV write)
  int padded_in;
  // padded_in 0: a non-rejected row left out of the K kept rows of its request
  // sets PE_ST_ROWS_RANGE (several layers need every row)
  int must_fit;
  uint32_t* status;
  int vec4;  // set by launch_rope_kv: four elements per load and store
};
int launch_rope_kv(const RopeArgs& a, int dtype, cudaStream_t st);

// ---------------------------------------------------------------- attention
struct AttnArgs {
  int B, K, H, G, hd, bs, max_blocks, num_blocks;
  int n_splits, split_len;
  // 1: the n_splits CTAs of one (request, KV head) are a thread-block cluster
  // and merge their partials in distributed shared memory (part_o / part_ml and
  // the combine kernel unused); 0: partials in global memory + combine kernel
  int cluster;
  const void* q;  // [B*K][H][hd]
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* seq_len;
  float* part_o;   // [n_splits][B*K][H][hd]     (bf16 path)
  float* part_ml;  // [n_splits][B*K][H][2]      (bf16 path)
  void* out;       // [B*K][H*hd]
  const float* sink;  // [H] per-head sink logit (natural units), nullable
  int k_min;          // seq_len below this is an input error (the draft depth K)
  uint32_t* status;
  // set by launch_attention for grids of several waves at head size 64: the longest-first unit
  // order (scratch after the partials); null: the 3-D grid (split, KV head, request)
  int2* order;
};
int attention_split_count(int B, int G, int max_blocks, int bs, int num_sms);
void plan_attention(int B, int G, int K, int H, int hd, int max_blocks, int bs, int num_sms,
                    int& n_splits, int& split_len, int& cluster);
size_t attention_scratch_bytes(int B, int K, int H, int hd, int n_splits);
int launch_attention(const AttnArgs& a, int dtype, cudaStream_t st);

// ---------------------------------------------------------------- argmax keys
// keys[0..n) = 0 (a kernel, so the LM head that follows can start early)
int launch_zero_keys(unsigned long long* keys, int n, cudaStream_t st);
// keys -> ids: out[i * stride] for i < n
int launch_argmax_finalize(const unsigned long long* keys, int n, int32_t* out, cudaStream_t st,
                           int stride = 1);

// ---------------------------------------------------------------- bounded-wait check
// one kernel whose bounded wait can never be satisfied: it records PE_ST_TIMEOUT
int launch_bounded_wait(uint32_t* status, cudaStream_t st);

}  // namespace pe
