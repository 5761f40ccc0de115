/*
 * pe_testing.h -- unit-test hooks of libpe: one drafter projection in isolation,
 * and the bounded device wait run out on purpose.
 *
 * Not part of the parallel-draft step.  It runs exactly the kernel the step runs
 * for one of the drafter's projections (tcgen05 GEMM for bf16, SIMT GEMM for
 * fp32) so tests can check that kernel alone against a matrix product.  Same
 * conventions as pe.h: device pointers owned by the caller, asynchronous on
 * `stream`, no allocation.
 */
#ifndef PE_TESTING_H
#define PE_TESTING_H

#include "pe.h"

#ifdef __cplusplus
extern "C" {
#endif

enum {
  PE_PROJ_FC = 0,     /* X [n][4d]   . w_fc^T   -> float [n][d]        */
  PE_PROJ_QKV = 1,    /* X [n][d]    . w_qkv^T  -> float [n][(H+2G)hd] */
  PE_PROJ_O = 2,      /* X [n][H hd] . w_o^T    -> float [n][d]        */
  PE_PROJ_SWIGLU = 3, /* silu(X w_gate^T) * (X w_up^T) -> dtype [n][I] */
  PE_PROJ_DOWN = 4,   /* X [n][I]    . w_down^T -> float [n][d]        */
  PE_PROJ_LM = 5,     /* X [n][d]    . w_lm^T   -> float [n][V]        */
  /* flags OR'ed into `which` */
  PE_PROJ_PERSISTENT = 0x100, /* never split K over a cluster: the persistent
                                 schedule with its tail split */
  PE_PROJ_PAIR = 0x200,       /* bf16 only: X holds n rows of high parts followed
                                 by n rows of low parts; the operand is hi + lo */
  PE_PROJ_PARTIAL = 0x400,    /* not with PE_PROJ_SWIGLU: each K split stores its
                                 partial sum, out = float [16][n][M] (split k at
                                 out + k*n*M; tiles past the split count are left
                                 as they were); the result is their sum */
  PE_PROJ_ARGMAX = 0x2000     /* PE_PROJ_LM only: the LM head with its argmax
                                 epilogue, as pe_argmax runs it: out = float
                                 logits [n][V]; the argmax of each row (int32 [n])
                                 is written to the workspace at byte offset
                                 PE_PROJ_ARGMAX_TOKENS_OFFSET(n) */
};

/* where PE_PROJ_ARGMAX leaves the row maxima' indices in the workspace */
#define PE_PROJ_ARGMAX_TOKENS_OFFSET(n) (256u + (((size_t)(n) * 8u + 255u) / 256u) * 256u)

/* Workspace bytes pe_test_projection needs for n_rows rows (0 on bad input). */
size_t pe_test_projection_workspace(const pe_handle* h, int which, int n_rows);

/* Run projection `which` over n_rows rows of X (the handle's dtype, row-major).
 * Returns PE_ERR_ARG / PE_ERR_UNSUPPORTED on bad input, PE_ERR_CUDA on a launch
 * failure.  The status word is the first 4 bytes of ws (pe_read_status). */
int pe_test_projection(pe_handle* h, int which, const void* X, int n_rows, void* out, void* ws,
                       size_t ws_bytes, void* stream);

/* Failure-detection check: one kernel whose bounded device wait (the mbarrier
 * wait every kernel of the step uses, limit 2 s) waits on a barrier that nothing
 * ever arrives on.  When the limit runs out the kernel ORs PE_ST_TIMEOUT into the
 * status word (the first 4 bytes of ws, at least 256 bytes, 16-byte aligned) and
 * returns; nothing faults and the context stays usable.  The caller clears the
 * word first (pe_read_status with clear set). */
int pe_test_bounded_wait(void* ws, size_t ws_bytes, void* stream);

/* Failure-detection check of the persistent decode layer (a bf16 one-layer step
 * of at most 16 rows): the byte of the step workspace that holds the count of
 * the layer's first kernel's completed launches within the step (uint32, zeroed
 * by pe_prepare_inputs).  A test that sets it far ahead after pe_prepare_inputs
 * makes that kernel's first grid barrier unreachable: its bounded wait runs out
 * (2 s), PE_ST_TIMEOUT goes into the status word and every CTA leaves. */
#define PE_TEST_DECODE_EPOCH_BYTE 112u

#ifdef __cplusplus
}
#endif
#endif /* PE_TESTING_H */
