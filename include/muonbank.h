/*
 * muonbank.h -- C ABI of libmuonbank.so: the Muon optimizer step over stacked
 * parameter banks on one NVIDIA GB300 (sm_103a).
 *
 * What one step computes, for every matrix X of a bank [batch, rows, cols]
 * independently (sources by page and section):
 *   S1  momentum   buf <- lerp(buf, g, 1-mu);  u <- lerp(g, buf, mu)
 *                  ("Muon Custom Sizing" write-up, record 2025-09-23, section 4,
 *                  second pass; Nesterov form named in the "UNetDoubleLr"
 *                  write-up, record 2024-11-10, optimizer section)
 *   S2  normalise  X0 = u / (||u||_F + 1e-7)  (the pages normalise by the
 *                  spectral norm; the Frobenius norm bounds it from above)
 *   S3  orientation: a tall matrix (rows > cols) iterates on X^T, which the
 *                  kernels realise as the swapped-operand form, with no copy
 *   S4  quintic Newton-Schulz, ns_steps times (5 by default):
 *                  A = X X^T;  B = b A + c A A;  X <- a X + B X,
 *                  (a, b, c) = (3.4445, -4.7750, 2.0315)
 *                  ("Muon Custom Sizing" write-up, section 2.3; Track-2
 *                  record 7 write-up, 2025-04-16, section 4.2)
 *                  Operands and stored A, B, X are bf16, with fp32
 *                  accumulation and fp32 epilogue arithmetic; matrices with
 *                  min(rows, cols) <= 64 run the whole iteration in fp32.
 *   S5  update     w32 = (w_bf16_bits << 16) | mantissa;
 *                  w32 <- w32 * (1 - lr*wd);  w32 <- w32 - lr*sqrt(max(1, rows/cols)) * v;
 *                  w_bf16_bits = w32 >> 16;  mantissa = w32 & 0xFFFF
 *                  (Track-2 record 7 write-up, section 4.1; effective lr and
 *                  decay from the "Muon Custom Sizing" write-up, section 4)
 *   S6  NorMuon (normuon_bank_step only; the "Unified zero-copy optimizer"
 *                  write-up, record 2026-01-18, names NorMuon but gives no
 *                  formula; this library reads it as): per row i of the
 *                  stored matrix q_i = mean_j v_ij^2, s_i <- beta2 s_i +
 *                  (1-beta2) q_i, v_ij <- v_ij / sqrt(max(s_i, 1e-10)), then
 *                  v is rescaled to its Frobenius norm before S5.
 *
 * Conventions shared by every entry point
 *   - Buffers are device pointers owned by the caller, row-major and
 *     contiguous: matrix k of a bank starts at k*rows*cols elements.  bf16
 *     tensors are passed as raw 16-bit patterns.  Every pointer must be
 *     16-byte aligned.
 *   - The library never allocates.  Scratch is a caller-provided device
 *     workspace of at least the size the *_workspace_bytes query returns;
 *     its contents need no initialisation and are overwritten.
 *   - Calls enqueue work on `cuda_stream` (a cudaStream_t; NULL = legacy
 *     default stream) and return without synchronising the host.
 *   - Return value: MB_OK (0) or a negative MB_ERR_* code.  Argument errors
 *     are detected before anything is enqueued.  A launch failure returns
 *     MB_ERR_CUDA (text from mb_last_cuda_error()).  A device-side fault
 *     detected while running (a bounded wait that expired) is latched in a
 *     per-device error word and returned by mb_sync_status().
 *   - Results are bit-identical from run to run (no float atomics).
 *   - In-place state (bank, mantissa, momentum, row state) must not alias
 *     any other argument.
 */
#ifndef MUONBANK_H_
#define MUONBANK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MB_OK = 0,
  MB_ERR_NULL = -1,          /* a required pointer is NULL */
  MB_ERR_SHAPE = -2,         /* batch/rows/cols <= 0, or a size past the limits of mb_shape */
  MB_ERR_ALIGN = -3,         /* a pointer is not 16-byte aligned */
  MB_ERR_NS_STEPS = -4,      /* ns_steps outside 0..16 */
  MB_ERR_WORKSPACE = -5,     /* workspace NULL or smaller than required */
  MB_ERR_CUDA = -6,          /* a CUDA runtime call or kernel launch failed */
  MB_ERR_TIMEOUT = -7,       /* a device-side bounded wait expired (from mb_sync_status) */
  MB_ERR_ARG = -8,           /* a scalar argument is not finite, or beta2/mu outside [0, 1] */
  MB_ERR_UNSUPPORTED = -9,   /* the current device is not sm_103 */
  MB_ERR_TOO_MANY = -10,     /* more banks than one call accepts */
  MB_ERR_SCRATCH_LIMIT = -11, /* mb_newton_schulz_noalloc: the shape needs more than its fixed scratch */
  MB_ERR_DEVICE = -12        /* a device-side consistency check failed (from mb_sync_status) */
};

/* One bank: `batch` matrices of rows x cols.  Limits (else MB_ERR_SHAPE): rows x cols
 * <= 2^30 elements per matrix, batch x rows x cols <= 2^40, batch x rows <= 2^30, and
 * batch x ceil(rows x cols / 8192) <= 2^30; the banks of one multi-bank call together
 * hold at most 2^30 matrices, 2^30 rows and 2^30 such 8192-element blocks. */
typedef struct {
  int32_t batch, rows, cols;
} mb_shape;

/* One bank of a multi-bank call (the launch sequence of a whole model step). */
typedef struct {
  void* bank;            /* bf16 [batch, rows, cols], updated in place */
  const void* grad;      /* bf16 [batch, rows, cols], read only */
  float* momentum;       /* fp32 [batch, rows, cols], updated in place */
  uint16_t* mantissa;    /* uint16 [batch, rows, cols], updated in place */
  float* row_state;      /* fp32 [batch, rows] NorMuon second moment; NULL unless normuon */
  mb_shape shape;
  void* bank_copy;       /* optional bf16 [batch, rows, cols]: the update also writes the new bank
                            here (for example for a download that overlaps the next step);
                            NULL: not written.  16-byte aligned, must not overlap any other
                            buffer of the call. */
} mb_bank_desc;

#define MB_MAX_BANKS 8

/* Bytes of workspace that muon_bank_step (normuon = 0) or normuon_bank_step
 * (normuon = 1) needs for `shape`. */
int mb_workspace_bytes(mb_shape shape, int normuon, size_t* out_bytes);

/* One full Muon step (S1-S5) over a bank.  lr and wd are the caller's values
 * with any per-parameter multipliers folded in; mu is the momentum of this
 * step (the caller applies any warm-up).  ns_steps = 0 skips S4 (v = X0). */
int muon_bank_step(void* bank_bf16, const void* grad_bf16, float* momentum_f32,
                   uint16_t* mantissa, mb_shape shape, float lr, float wd, float mu,
                   int ns_steps, void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Muon step with the NorMuon per-row normalisation (S1-S4, S6, S5).
 * row_state_f32 is [batch, rows], updated in place; beta2 in [0, 1]. */
int normuon_bank_step(void* bank_bf16, const void* grad_bf16, float* momentum_f32,
                      uint16_t* mantissa, float* row_state_f32, mb_shape shape, float lr,
                      float wd, float mu, float beta2, int ns_steps, void* workspace,
                      size_t workspace_bytes, void* cuda_stream);

/* Workspace for muon_multi_step over `n_banks` descriptors. */
int mb_multi_workspace_bytes(const mb_bank_desc* banks, int n_banks, int normuon,
                             size_t* out_bytes);

/* One step over up to MB_MAX_BANKS banks with shared hyperparameters, as one
 * launch sequence: the element-wise stages run once over all banks and the
 * Newton-Schulz GEMMs of all large banks share each launch.  normuon selects
 * S6 for every bank (each then needs row_state).  The `banks` array is read on
 * the host during the call only. */
int muon_multi_step(const mb_bank_desc* banks, int n_banks, float lr, float wd, float mu,
                    int normuon, float beta2, int ns_steps, void* workspace,
                    size_t workspace_bytes, void* cuda_stream);

/* Options of muon_multi_step_ex.  Both move a pass over the step's elements into the
 * epilogue of the last Newton-Schulz GEMM (the tensor-core kernel then launches a second
 * instantiation that carries this code); both were measured and are off by default:
 *   MB_STEP_FUSE_UPDATE    without NorMuon: S5 runs in that epilogue on banks with
 *                          min(rows, cols) > 64 and cols a multiple of 8 (with at least 3
 *                          Newton-Schulz steps), reading v as it is stored; the separate
 *                          update pass then covers only the other banks.  Same bits as the
 *                          default path.  On the GPT-2-small step it made the step slower
 *                          (1.35 vs 1.14 ms on one GB300): the epilogue, already the
 *                          Newton-Schulz kernel's bound, waits on the bank and mantissa loads.
 *   MB_STEP_FUSE_ROWSTATS  with NorMuon: the row sums of v^2 come from that epilogue (per
 *                          32-column chunk, added in a fixed order by the row-scale pass)
 *                          instead of a pass that reads v again.  Same results up to fp32
 *                          summation order; measured even on the GPT-2-medium step.
 * Unknown bits: MB_ERR_ARG.  v is still stored in the workspace (mb_workspace_views). */
#define MB_STEP_FUSE_UPDATE 1u
#define MB_STEP_FUSE_ROWSTATS 2u
int muon_multi_step_ex(const mb_bank_desc* banks, int n_banks, float lr, float wd, float mu,
                       int normuon, float beta2, int ns_steps, unsigned flags, void* workspace,
                       size_t workspace_bytes, void* cuda_stream);

/* muon_multi_step with each bank's hyperparameters read from device memory when
 * the step runs, so that a captured CUDA graph of the step can be replayed with
 * new values ("Unified zero-copy optimizer" write-up, section 4: all banks' step
 * scalars in one fp32 device buffer, uploaded once per step, read by the graph).
 *   scalars_dev : device pointer, 16-byte aligned, n_banks x {lr, wd, mu, beta2}
 *                 fp32 (beta2 only read with normuon); the caller owns it and may
 *                 rewrite it between steps (stream-ordered with the step).
 * Results are bit-identical to muon_multi_step with the same values.  Values
 * are checked on the device: a non-finite value, or mu or beta2 outside [0, 1],
 * makes mb_sync_status return MB_ERR_ARG and leaves the step's outputs undefined.
 * Host-side errors as for muon_multi_step; MB_ERR_NULL / MB_ERR_ALIGN for
 * scalars_dev.  One more (single-block) launch than muon_multi_step. */
int muon_multi_step_dev(const mb_bank_desc* banks, int n_banks, const float* scalars_dev,
                        int normuon, int ns_steps, void* workspace, size_t workspace_bytes,
                        void* cuda_stream);

/* ---- single stages, for callers that run them separately (and for tests) ---- */

/* S1 only: momentum in place and u (bf16 [batch, rows, cols], dense) out. */
int mb_momentum(const void* grad_bf16, float* momentum_f32, void* u_bf16, mb_shape shape,
                float mu, void* cuda_stream);

/* S2-S4 only: v = NS(u / (||u||_F + 1e-7)) per matrix, v bf16 dense [batch, rows, cols].
 * Uses the muon_bank_step workspace (normuon = 0). */
int mb_newton_schulz(const void* u_bf16, void* v_bf16, mb_shape shape, int ns_steps,
                     void* workspace, size_t workspace_bytes, void* cuda_stream);

/* mb_newton_schulz with a coefficient schedule: step i uses (a, b, c) =
 * coeffs[3i], coeffs[3i+1], coeffs[3i+2] instead of the quintic (3.4445, -4.7750,
 * 2.0315) that every other call uses for every step ("Muon Custom Sizing",
 * section 2.3).  For per-iteration schedules such as the Polar Express
 * orthogonalisation named in the "Unified zero-copy optimizer" write-up (section 4),
 * whose coefficients the pages do not print.  coeffs: host array of 3 * ns_steps
 * finite floats, read during the call.  MB_ERR_NULL / MB_ERR_ARG for coeffs, other
 * errors as mb_newton_schulz.  The bf16 tolerance of the result depends on the schedule. */
int mb_newton_schulz_coeffs(const void* u_bf16, void* v_bf16, mb_shape shape, int ns_steps,
                            const float* coeffs, void* workspace, size_t workspace_bytes,
                            void* cuda_stream);

/* S2-S4 like mb_newton_schulz, for callers that cannot allocate device memory.
 *
 * Not part of the method on the speedrun pages (they have no counterpart);
 * it exists for callers that may not call cudaMalloc: code running inside a
 * memory pool or allocator callback, a host whose allocator is owned by
 * another framework, or a process that must not grow its device footprint
 * after start-up.  Such callers cannot provide the workspace that
 * mb_newton_schulz needs, so this variant uses a scratch array that the
 * library holds as a fixed device global of MB_NOALLOC_SCRATCH_BYTES on every
 * GPU that loads it, for the life of the process.  The caller still passes u
 * and v (bf16 dense [batch, rows, cols]).
 *   - Returns MB_ERR_SCRATCH_LIMIT, and enqueues nothing, when the shape needs
 *     more scratch than that (mb_workspace_bytes(shape, 0) is the need).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array, and it keeps the previous
 *     call's contents.  Nothing in it has to start at zero (every byte is
 *     written before it is read).  Calls that overlap on the GPU, from
 *     different streams or threads, race on it: serialise them. */
#define MB_NOALLOC_SCRATCH_BYTES (32u << 20)
int mb_newton_schulz_noalloc(const void* u_bf16, void* v_bf16, mb_shape shape, int ns_steps,
                             void* cuda_stream);

/* S5 only, given v (bf16 dense). */
int mb_update(void* bank_bf16, uint16_t* mantissa, const void* v_bf16, mb_shape shape,
              float lr, float wd, void* cuda_stream);

/* S6 then S5, given v (bf16 dense); uses the normuon_bank_step workspace. */
int mb_normuon_update(void* bank_bf16, uint16_t* mantissa, const void* v_bf16,
                      float* row_state_f32, mb_shape shape, float lr, float wd, float beta2,
                      void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Where a finished muon_bank_step / normuon_bank_step left u (the bf16 NS
 * input) and v (the bf16 NS output) inside its workspace: byte offsets from
 * the workspace start and the row pitch in elements (>= cols); matrix k of
 * each starts at k * rows * pitch elements. */
int mb_workspace_views(mb_shape shape, int normuon, int ns_steps, size_t* u_offset,
                       size_t* v_offset, size_t* row_pitch);

/* Synchronises `cuda_stream`, then returns and clears this device's latched
 * device-side status (MB_OK, MB_ERR_TIMEOUT, MB_ERR_ARG for a bad scalar read
 * by muon_multi_step_dev, or MB_ERR_DEVICE), or MB_ERR_CUDA. */
int mb_sync_status(void* cuda_stream);

/* Runs the bounded-wait primitive of the kernels against an mbarrier that
 * nothing completes, with a limit of `limit_us` microseconds; the kernel gives
 * up, latches MB_ERR_TIMEOUT and returns.  For testing failure detection. */
int mb_selftest_timeout(unsigned limit_us, void* cuda_stream);

/* ---- measurement hooks ---- */

/* Number of kernels this host thread has launched through the library so far. */
uint64_t mb_launch_count(void);

/* Stage labels of the timing marks. */
enum {
  MB_MARK_BEGIN = 0,      /* start of a step (or stage call) */
  MB_MARK_MOMENTUM = 1,   /* after S1 (and the u^2 partial sums) */
  MB_MARK_SCALE = 2,      /* after the per-matrix 1/(||u||+eps) */
  MB_MARK_SMALL_NS = 3,   /* after the fp32 Newton-Schulz of small matrices */
  MB_MARK_NS_GEMM = 4,    /* after the tensor-core Newton-Schulz launch (all steps) */
  MB_MARK_NS0 = 5,        /* after the ns_steps = 0 scaling, or the copy-out of a stage call */
  MB_MARK_ROWSTATS = 6,   /* after the NorMuon row statistics */
  MB_MARK_UPDATE = 7      /* after S5 */
};

/* Starts recording a CUDA event on the launching stream at every stage
 * boundary of the following calls made by this host thread, up to
 * `max_marks` marks (events are created here; no device memory is allocated). */
int mb_timing_begin(int max_marks);

/* Stops recording, synchronises the events and returns up to `cap` marks:
 * labels[i] (MB_MARK_*) and ms[i] = milliseconds from the previous mark to
 * mark i (0 for MB_MARK_BEGIN).  *n_marks receives the number recorded. */
int mb_timing_end(int cap, int* labels, float* ms, int* n_marks);

/* Static text of a status code; the last CUDA error message of this thread. */
const char* mb_status_string(int status);
const char* mb_last_cuda_error(void);

/* Library version, (major << 16) | minor. */
int mb_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MUONBANK_H_ */
