// Internal interfaces between the C ABI (mb_api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mb {

constexpr int MAX_BANKS = 8;       // banks per element-wise launch
constexpr int SMALL_M = 64;        // min(rows, cols) <= SMALL_M: fp32 SIMT Newton-Schulz
constexpr int MAX_NS_STEPS = 16;   // Newton-Schulz steps one call accepts

// Elements handled by one block of the element-wise kernels (per matrix chunk).
constexpr int EW_THREADS = 256;
constexpr int EW_CHUNK = EW_THREADS * 8 * 4;

// ---------------------------------------------------------------- element-wise stages

struct EwBank {
  const uint16_t* src;     // K1: grad (momentum) or u (pack); K3: unused
  float* mom;              // K1 momentum (null in pack mode)
  uint16_t* bank;          // K3 weight bf16 bits
  uint16_t* mant;          // K3 mantissa
  uint16_t* bank_copy;     // K3: optional second destination of the updated bf16 bank (null: none)
  uint16_t* xout;          // K1: u destination (pitch ld); ns0/unpack: destination
  const uint16_t* xin;     // K3/ns0/unpack: source (pitch ld)
  const float* rowscale;   // K3 NorMuon per-row factor (null otherwise)
  float* partials;         // K1: per-chunk sum of u^2, [batch * P] (null = skip)
  const float* scale;      // ns0: per-matrix 1/(||u||+eps)
  int batch, rows, cols, ld, out_ld;
  int P;                   // chunks per matrix
  int block_begin;         // first block of this bank in the launch
  float decay, neg_lr;     // K3: 1 - lr*wd, -lr*sqrt(max(1, rows/cols))
  const float* dscal;      // this bank's scalars in device memory (DSCAL_* order), or null: use the fields above
};

// Derived per-bank scalars of a step whose hyperparameters are read from device
// memory (muon_multi_step_dev), in the workspace: the values the host forms in
// double for the by-value calls, formed the same way by scalars_kernel.
enum DerivedScalar { DSCAL_MU = 0, DSCAL_OMM, DSCAL_DECAY, DSCAL_NEG_LR, DSCAL_BETA2, DSCAL_COUNT = 8 };
struct ScalarBank {
  const float* src;        // caller's {lr, wd, mu, beta2} of this bank
  float* dst;              // DSCAL_COUNT derived values
  double shape_factor;     // sqrt(max(1, rows / cols)), formed on the host
};
struct ScalarParams {
  ScalarBank b[MAX_BANKS];
  int nb, normuon;
  int* status;
};

struct EwParams {
  EwBank b[MAX_BANKS];
  int nb;
  int total_blocks;
  float mu, omm;           // K1: momentum and 1 - mu (formed in double on the host)
  int* status;
};

// Per-matrix scale s = 1/(sqrt(sum partials) + eps).
struct ScaleBank {
  const float* partials;
  float* scale;
  int batch, P, mat_begin;
};
struct ScaleParams {
  ScaleBank b[MAX_BANKS];
  int nb, total_mats;
};

// fp32 SIMT Newton-Schulz for small matrices: one block per matrix.
struct SmallBank {
  const uint16_t* x0;   // u, bf16, pitch ld
  float* xf0;           // fp32 scratch [batch, rows, cols]
  float* xf1;
  uint16_t* out;        // bf16 result, pitch ld
  const float* scale;
  int batch, rows, cols, ld;
  int block_begin;
};
struct SmallParams {
  SmallBank b[MAX_BANKS];
  int nb, total_blocks, steps;
  float ca[MAX_NS_STEPS], cb[MAX_NS_STEPS], cc[MAX_NS_STEPS];   // (a, b, c) of each step
};

// NorMuon row statistics and scales.
struct RowBank {
  const uint16_t* v;    // NS output, pitch ld
  float* q;             // per-row sum of v^2 [batch * rows]
  const float* rowsq;   // or, from the Newton-Schulz epilogue: sums per 32-column chunk [batch][nchunk][rows]
  int nchunk;
  float* state;         // row second moment [batch * rows] (in place)
  float* rowscale;      // per-row factor [batch * rows]
  int batch, rows, cols, ld;
  int row_begin;        // prefix over rows (KN1) ...
  int mat_begin;        // ... and over matrices (KN2)
  const float* dscal;   // derived scalars in device memory, or null: use RowParams::beta2
};
struct RowParams {
  RowBank b[MAX_BANKS];
  int nb, total_rows, total_mats;
  float beta2;
};

// ---------------------------------------------------------------- Newton-Schulz GEMMs

enum GemmEpi { EPI_GRAM = 0, EPI_POLY = 1, EPI_APPLY = 2 };   // the three GEMM phases of one step

// What the last step's APPLY epilogue of a bank does beyond storing v:
//   FIN_UPDATE  S5 on the output in place: the bank and mantissa (and the optional bank copy)
//               are read, updated with the bf16-rounded v and written back by that epilogue;
//   FIN_ROWSQ   NorMuon: the sums of v^2 of each row over each 32-column chunk, per matrix,
//               into rowsq [batch][nchunk][rows] (chunk-major), for the row-scale kernel.
enum FinMode { FIN_NONE = 0, FIN_UPDATE = 1, FIN_ROWSQ = 2 };

constexpr int MAX_NS_BANKS = 4;     // large banks per fused Newton-Schulz launch

// One large bank in the fused Newton-Schulz launch.  x[0] holds u; the
// iterates X_1, X_2, ... alternate between x[1] and x[2].
// Every operand tile of one 64-deep k-block is a single TMA box: K-major boxes
// of 128 rows, and MN-major boxes of 2 chunks of 64 columns through a 4-D view
// {64 columns, rows, row pitch / 64 chunks, matrix} of an X buffer (large banks
// pitch their X buffers to a multiple of 64 columns for it).
struct NsBank {
  CUtensorMap xk[3];                // X buffers, K-major boxes of 128 rows x 64
  CUtensorMap xmn2[3];              // X buffers, MN-major boxes of 64 K rows x 128 columns
  CUtensorMap ak, bk;               // A and B, K-major boxes of 128 rows x 64
  CUtensorMap st_x[3], st_a, st_b;  // 32x32 boxes (64-byte swizzle): the epilogues' stores, and their inputs
  const float* scale;               // per-matrix 1/(||u||_F + eps)
  unsigned* done;                   // completion counters [batch][MAX_NS_STEPS][3], zeroed before launch
  int batch, rows, cols, m, n, tall;
  int T, sym_pairs;                 // 128-blocks per side of A; pair tasks per matrix of GRAM and POLY
  int tn, apply_pairs;              // 256-wide column tiles and pair tasks per matrix of APPLY
  // the last step's APPLY epilogue (FinMode); FIN_UPDATE needs cols % 8 == 0 (16-byte row pieces)
  int fin, store_v;                 // store_v = 0: the last APPLY writes no v (FIN_UPDATE only)
  uint16_t* w;                      // FIN_UPDATE: bank bf16 bits [batch, rows, cols], in place
  uint16_t* mant;                   //             mantissa, in place
  uint16_t* w_copy;                 //             optional second destination of the bank, or null
  float decay, neg_lr;              //             1 - lr*wd, -lr*sqrt(max(1, rows/cols))
  const float* dscal;               //             derived scalars in device memory, or null
  float* rowsq;                     // FIN_ROWSQ: [batch][nchunk][rows] partial sums of v^2
  int nchunk;                       //            ceil(cols / 32)
};

struct NsParams {
  NsBank bank[MAX_NS_BANKS];
  int nbank, steps;
  // one step's tasks come as (bank, phase) segments in this order; seg_begin[nseg] is the step's size
  int nseg;
  int seg_begin[3 * MAX_NS_BANKS + 1];
  unsigned char seg_bank[3 * MAX_NS_BANKS], seg_ph[3 * MAX_NS_BANKS];
  int tasks_per_iter, total_tasks;
  unsigned* next_task;              // dynamic scheduler, zeroed before launch
  float ca[MAX_NS_STEPS], cb[MAX_NS_STEPS], cc[MAX_NS_STEPS];   // (a, b, c) of each step
  int* status;
};

// ---------------------------------------------------------------- launchers (return cudaError_t)

cudaError_t launch_k1(const EwParams& p, bool momentum, cudaStream_t s);
cudaError_t launch_scale(const ScaleParams& p, cudaStream_t s);
cudaError_t launch_ns0(const EwParams& p, cudaStream_t s);
cudaError_t launch_unpack(const EwParams& p, cudaStream_t s);
// Shared memory the in-shared-memory fp32 NS needs for one rows x cols matrix;
// banks up to SMALL_SMEM_MAX use it, larger ones run through the workspace.
constexpr int SMALL_SMEM_MAX = 200 * 1024;
long long small_ns_smem_bytes(int rows, int cols);
cudaError_t launch_small_ns(const SmallParams& p, bool in_smem, cudaStream_t s);
cudaError_t launch_row_sumsq(const RowParams& p, cudaStream_t s);
cudaError_t launch_row_scale(const RowParams& p, cudaStream_t s);
cudaError_t launch_k3(const EwParams& p, bool normuon, cudaStream_t s);
cudaError_t launch_scalars(const ScalarParams& p, cudaStream_t s);
cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t s);
cudaError_t launch_ns_fused(const NsParams& p, cudaStream_t s);       // plain or with FinModes, as the banks ask
cudaError_t launch_ns_fused_fin(const NsParams& p, cudaStream_t s);   // the instantiation with FinModes

}  // namespace mb
