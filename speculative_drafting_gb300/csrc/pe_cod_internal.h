// Shared by the two COD sources: launch shapes, the workspace header, the
// depth bound, the sequence-length clamp and the host-side argument checks.
#ifndef PE_COD_INTERNAL_H
#define PE_COD_INTERNAL_H

#include "pe_common.cuh"
#include "pe_internal.h"

namespace pe {

constexpr int kMaskThreads = 256;
constexpr int kMaskWarps = kMaskThreads / 32;
constexpr int kWsHeader = 256;  // status word, then the place table
constexpr int kMaxD = PE_COD_MAX_DEPTH;

PE_DEV int clamp_len(int L, int S_max) { return L < 0 ? 0 : (L > S_max ? S_max : L); }

}  // namespace pe

// Checks both COD calls share (sizes, depth, workspace, seq_len); PE_OK or an error code.
int cod_common_args(int B, int S_max, int n_depth, const void* seq_len, void* ws, size_t ws_bytes);

#endif  // PE_COD_INTERNAL_H
