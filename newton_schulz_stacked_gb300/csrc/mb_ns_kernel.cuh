// Batched Newton-Schulz iteration on the sm_103a tensor cores (tcgen05 + TMEM,
// operands staged by TMA with 128-byte swizzle), all steps in one launch: the
// kernel template, instantiated plain in mb_ns_gemm.cu and with the last-step
// modes (FinMode) in mb_ns_gemm_fin.cu.
//
// One quintic step ("Muon Custom Sizing" write-up, section 2.3; Track-2
// record 7 write-up, section 4.2) is three GEMM phases per matrix:
//   GRAM   A  = alpha * X X^T         (alpha = s^2 on the first step, s = 1/(||u||+eps))
//   POLY   B' = a I + b A + c A A     (A symmetric, so A A = A A^T)
//   APPLY  X' = beta B' X             (beta = s on the first step)
// so that a X + b A X + c A^2 X needs no X in APPLY's epilogue: a I rides in the stored bf16
// B'.  The second step also adds a times the first iterate's bf16 residual (stored by the
// first step's APPLY), so that its a X term sees X_1 to ~16 bits.  A tall slice (rows > cols)
// stays in its stored orientation and runs the swapped-operand form A = X^T X,
// X' = beta X B'; the difference is only which operand tiles are K-major and which MN-major.
//
// CTA pairs.  The kernel runs in clusters of two CTAs (one per SM) that compute
// one 256 x nt output tile (nt = 128 or 256) with M = 256 tcgen05 MMAs
// (cta_group::2): CTA r holds tile rows 128r .. 128r+127 of the A operand and
// half of the B operand's nt rows, and its TMEM receives its 128 rows x all nt
// columns.  Each SM therefore stages 32 KB of operands per 64-deep k-block
// instead of 48 KB for a 128 x 256 tile alone: a third less L2-to-SM traffic,
// and five stages in flight where four fitted before, with room left for the
// epilogue's input ring.
//
// A and B are symmetric: GRAM and POLY compute only the 256 x 256 tiles (2 x 2
// aligned 128-blocks) that touch the upper triangle.  Each block above the
// diagonal is stored twice, directly and mirrored, so the next phase reads a
// full matrix; a block on the diagonal is made symmetric before its store, and
// the one block below the diagonal of a diagonal tile is computed but not stored.
//
// Scheduling.  The work of all steps is one list of pair tasks (a 256-row
// output tile of one phase of one matrix), ordered by step, then by (bank,
// phase) segment in the order the host gives (any order that puts each bank's
// GRAM before its POLY before its APPLY), then matrix and tile.  The even CTA
// of each pair claims tasks from a global counter and hands them to both CTAs.
// A task's loads first wait until every tile of the previous phase of the same
// matrix has been stored (per-matrix completion counters, release/acquire at
// GPU scope), so phases overlap across matrices and there is no launch
// boundary between them.  Every task depends only on earlier tasks and all
// pairs are resident, so the earliest unfinished task can always run; each
// wait is bounded all the same.
//
// CTA roles (11 warps, both CTAs unless noted):
//   warp 10 lane 0: (even CTA) scheduler: claims the next task, decodes it and
//                   waits until its inputs are stored, one task ahead of the
//                   producer, and writes the decoded task into both CTAs' ring
//                   of task records (the odd CTA's through distributed shared
//                   memory); (odd CTA) relay: once every reader of a record in
//                   the odd CTA has taken it, tells the scheduler with one
//                   cluster-scope arrival
//   warp 0 lane 0 : TMA producer of a STAGES-deep ring of (A 128x64, B-half
//                   128x64) bf16 tiles, one TMA box per operand and k-block (a
//                   producer thread pays about as much per TMA instruction as an
//                   MMA of one 16-deep slice takes); the bytes of both CTAs
//                   complete on the even CTA's stage barrier
//   warp 1        : allocates 512 TMEM columns in both CTAs = two 256-column
//                   fp32 accumulators; (even CTA) lane 0 issues the MMAs and
//                   releases each stage in both CTAs with a multicast commit
//   warps 2..9    : epilogue of the CTA's own 128 rows, two warps per 32-lane
//                   TMEM quadrant (each takes half the columns); task k's
//                   epilogue runs under task k+1's MMAs; its input (A for POLY's
//                   b A, X_1's residual in the second step's APPLY) arrives
//                   by TMA in 32x32 boxes through a two-slot ring refilled as each
//                   chunk is taken, and its results leave through shared memory by
//                   TMA bulk stores; a chunk moves as 8x8 matrices in MMA-fragment
//                   order (16-lane TMEM loads, ldmatrix, stmatrix and, for the
//                   mirror of a symmetric chunk, stmatrix.trans)
#pragma once

#include <atomic>

#include "mb_device.cuh"
#include "mb_internal.h"

namespace mb {

namespace {

constexpr int BM = 128;                      // rows of a tile per CTA
constexpr int BK = 64;
constexpr int STAGES = 5;
constexpr int A_TILE_BYTES = BM * BK * 2;    // 16 KB
constexpr int BH_TILE_BYTES = 128 * BK * 2;  // 16 KB: this CTA's half of a 256-row B operand
constexpr int STAGE_BYTES = A_TILE_BYTES + BH_TILE_BYTES;
constexpr int TILE_SMEM = STAGES * STAGE_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int EPI_BUF_BYTES = 4096;          // per epilogue warp: 32x32 bf16 chunk + its transpose
constexpr int EPI_SMEM = EPI_WARPS * EPI_BUF_BYTES;
constexpr int IN_SLOTS = 2;                  // per epilogue warp: input chunks in flight
constexpr int IN_BOX_BYTES = 32 * 32 * 2;    // one 32x32 bf16 input chunk
constexpr int IN_SMEM = EPI_WARPS * IN_SLOTS * IN_BOX_BYTES;
constexpr int TASK_SLOTS = 4;                // claimed tasks in flight inside a pair
// threads that read a task record and arrive on their own CTA's slot_empty barrier: in the
// even CTA its producer, the MMA issuer, its epilogue warps and the odd CTA's relay; in the
// odd CTA its producer and epilogue warps
constexpr int SLOT_READERS_EVEN = 1 + 1 + EPI_WARPS + 1;
constexpr int SLOT_READERS_ODD = 1 + EPI_WARPS;
constexpr int GEMM_SMEM = TILE_SMEM + EPI_SMEM + IN_SMEM + 1024 /* alignment slack */ + 768 /* barriers, slots */;
static_assert(GEMM_SMEM <= 232448, "shared memory per CTA");
constexpr int SCHED_WARP = 2 + EPI_WARPS;
constexpr int GEMM_THREADS = 32 * (3 + EPI_WARPS);
constexpr uint32_t ACC_COLS = 256;           // one accumulator
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;

// ---------------------------------------------------------------- tasks

// One pair task, as the scheduler hands it over (t < 0: no more tasks).  The
// CTA of pair rank r computes rows m0 + 128 r .. m0 + 128 r + 127.
struct Task {
  int t;                 // task index
  int it, ph, bi, mat;   // step, phase, bank, matrix
  int m0, n0, nt;        // output tile origin (of the pair) and width (128 or 256)
};

__device__ __forceinline__ int iterate_buffer(int k) { return k == 0 ? 0 : 1 + ((k - 1) & 1); }

__device__ __forceinline__ void decode_task(const NsParams& P, int t, Task& k) {
  k.t = t;
  k.it = t / P.tasks_per_iter;
  int r = t - k.it * P.tasks_per_iter;
  int g = 0;
  while (g + 1 < P.nseg && r >= P.seg_begin[g + 1]) ++g;
  k.bi = P.seg_bank[g];
  k.ph = P.seg_ph[g];
  r -= P.seg_begin[g];
  const NsBank& B = P.bank[k.bi];
  k.m0 = k.n0 = 0;
  k.nt = 128;
  if (k.ph != EPI_APPLY) {
    // block-row pair q (128-blocks 2q, 2q+1) takes the block-column pairs p = q .. P2-1
    k.mat = r / B.sym_pairs;
    r -= k.mat * B.sym_pairs;
    const int P2 = (B.T + 1) >> 1;
    for (int q = 0; q < P2; ++q) {
      const int c = P2 - q;
      if (r < c) {
        const int p = q + r;
        k.m0 = 2 * q * BM;
        k.n0 = 2 * p * BM;
        k.nt = (2 * p + 1 < B.T) ? 256 : 128;
        return;
      }
      r -= c;
    }
  } else {
    k.mat = r / B.apply_pairs;
    r -= k.mat * B.apply_pairs;
    const int tm2 = r / B.tn, tj = r - tm2 * B.tn;
    const int N = B.tall ? B.m : B.n;
    k.m0 = 2 * tm2 * BM;
    k.n0 = tj * 256;
    k.nt = (N - k.n0 > 128) ? 256 : 128;
  }
}

// Tiles (one per CTA of a pair task) per matrix of a phase: what its completion counter reaches.
__device__ __forceinline__ int phase_tiles(const NsBank& B, int ph) {
  return 2 * (ph == EPI_APPLY ? B.apply_pairs : B.sym_pairs);
}

__device__ __forceinline__ unsigned* done_counter(const NsBank& B, int mat, int it, int ph) {
  return B.done + (static_cast<size_t>(mat) * MAX_NS_STEPS + it) * 3 + ph;
}

// Operands of a task's GEMM in one CTA of the pair: each is one box per k-block
// of 128 rows (K-major) or 128 columns (MN-major).  A CTA's half of a 128-wide B
// operand is 64 rows or columns; its box then also carries 64 that are not read.
struct Operands {
  const CUtensorMap* a;
  const CUtensorMap* b;
  int a_mn, b_mn, K;
};

__device__ __forceinline__ Operands task_operands(const NsBank& B, const Task& k) {
  const int cur = iterate_buffer(k.it);
  Operands o;
  if (k.ph == EPI_GRAM) {
    o.a = o.b = B.tall ? &B.xmn2[cur] : &B.xk[cur];   // A = X^T X (columns of X) or X X^T (rows)
    o.a_mn = o.b_mn = B.tall;
    o.K = B.n;
  } else if (k.ph == EPI_POLY) {
    o.a = o.b = &B.ak;
    o.a_mn = o.b_mn = 0;
    o.K = B.m;
  } else {
    if (!B.tall) {       // X' = B' X: rows of B' (K-major), X as MN-major tiles
      o.a = &B.bk;
      o.b = &B.xmn2[cur];
      o.a_mn = 0;
      o.b_mn = 1;
    } else {             // X' = X B': rows of X and of B', both K-major
      o.a = &B.xk[cur];
      o.b = &B.bk;
      o.a_mn = 0;
      o.b_mn = 0;
    }
    o.K = B.m;
  }
  return o;
}

// In a 256-wide tile on the diagonal of a symmetric phase (A = X X^T or X^T X, and A A with
// A symmetric), each CTA's half of the B operand holds the same rows, in the same layout, as
// its A tile: the producer loads only A and the MMAs read B from there.
__device__ __forceinline__ bool b_is_a(const Task& k) { return k.ph != EPI_APPLY && k.m0 == k.n0 && k.nt == 256; }

// ---------------------------------------------------------------- cross-CTA completion

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's generic-proxy view of global memory with its async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Waits (bounded) until *ctr >= target.
__device__ __forceinline__ bool wait_counter(const unsigned* ctr, unsigned target, const volatile int* abort) {
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(128);
    if (ld_acquire(ctr) >= target) return true;
    if ((i & 15u) == 0u && (*abort || globaltimer_ns() - t0 > WAIT_LIMIT_NS)) return false;
  }
}

// The phase a task reads from; false when it reads only the step's input u.
__device__ __forceinline__ bool dependency(const Task& k, int& dit, int& dph) {
  if (k.ph == EPI_GRAM) {
    if (k.it == 0) return false;
    dit = k.it - 1;
    dph = EPI_APPLY;
  } else {
    dit = k.it;
    dph = k.ph - 1;
  }
  return true;
}

// ---------------------------------------------------------------- epilogue

// Byte offset of 16-byte chunk `chunk` of row `row` in a [32][32] bf16 staging
// buffer laid out as the TMA 64-byte swizzle expects (address bits [4,6) XOR
// bits [7,9)): the eight 16-byte rows of an 8x8 matrix (ldmatrix / stmatrix) then hit
// distinct banks, and so do row-wise 16-byte accesses of a warp.
__device__ __forceinline__ uint32_t sw64(int row, int chunk) {
  return static_cast<uint32_t>(row * 64 + 16 * (chunk ^ ((row >> 1) & 3)));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return bf16_bits_to_float(w & 0xFFFFu); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return bf16_bits_to_float(w >> 16); }

struct EpiJob {
  const CUtensorMap* st;   // store map of the output
  // APPLY only: the first step also stores the bf16 residual of X_1 (st_lo), and the
  // second step's input adds it back so that its a*X_1 term uses X_1 to ~16 bits
  const CUtensorMap* st_lo;
  int M, N, sym, mat, m0, n0, nt;
  int it;                  // Newton-Schulz step: picks its (a, b, c)
  float alpha;
  int bi;                  // bank: the last step's APPLY reads its FinMode fields from P
};

// LO (APPLY only): 0 plain; LO_WRITE also stores the bf16 residual of the output (first
// step); LO_READ adds a times the residual stored by the first step (second step).
constexpr int LO_WRITE = 1, LO_READ = 2;

// Non-blocking: whether the phase with the given parity has completed (acquire at cluster scope).
__device__ __forceinline__ bool mbar_test_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Where one epilogue warp's input of a task comes from: chunk c is the 32x32 box at
// (col0 + 32 c, row0) of matrix `mat` of A (POLY) or of X_1's residual (the second step's
// APPLY), read through the map it was stored with (64-byte swizzle, so a lane reading its
// own row of the box hits distinct banks).  GRAM and the other APPLY steps read none (nch 0).
// Boxes reaching past the matrix read zeros.
struct InSrc {
  const CUtensorMap* map;
  int row0, col0, mat, nch;
  __device__ __forceinline__ int units() const { return nch; }
};

__device__ __forceinline__ InSrc input_of(const NsParams& P, const Task& tk, int row_base, int half) {
  InSrc s{nullptr, 0, 0, 0, 0};
  if (tk.t < 0 || tk.ph == EPI_GRAM || (tk.ph == EPI_APPLY && tk.it != 1)) return s;
  const NsBank& B = P.bank[tk.bi];
  s.map = tk.ph == EPI_POLY ? &B.st_a : &B.st_x[2];
  s.row0 = tk.m0 + row_base;
  s.col0 = tk.n0 + half * (tk.nt >> 1);
  s.mat = tk.mat;
  s.nch = tk.nt >> 6;   // (nt / 2) columns in 32-column chunks
  return s;
}

// One epilogue warp's input ring: IN_SLOTS shared buffers of one 32x32 box (a unit) each,
// refilled by TMA as soon as the epilogue has taken a chunk's units into registers, so the
// next units load under the chunk's work.  Once a task's units are all issued, the ring
// runs on into the next task's as soon as that task's record is published (a
// non-blocking test: the next task may depend on this one).  The counters are
// warp-uniform; lane 0 issues.
struct InFeed {
  uint8_t* buf;            // IN_SLOTS x IN_BOX_BYTES
  uint64_t* full;          // IN_SLOTS barriers: lane 0's expect_tx arrival, then the bytes
  const Task* rec;         // the task records ...
  uint64_t* slot_full;     // ... and their barriers
  uint32_t k;              // the task this warp is working on
  uint32_t issued, used;   // units issued and consumed so far
  InSrc cur, nxt;          // the inputs of task k and task k + 1
  int cur_iss, nxt_iss;    // how many of their units are issued
  bool nxt_known;
  int row_base, half;      // this warp's rows (CTA rank and quadrant) and column half
};

// Unit (chunk) u of a task's input.
__device__ __forceinline__ void in_issue(InFeed& F, const InSrc& s, int u, int lane) {
  if (lane == 0) {
    const uint32_t slot = F.issued % IN_SLOTS;
    mbar_expect_tx(&F.full[slot], IN_BOX_BYTES);
    tma_load_3d(F.buf + slot * IN_BOX_BYTES, s.map, &F.full[slot], s.col0 + 32 * u, s.row0, s.mat);
  }
  ++F.issued;
}

// Issues input units while the ring has room: the rest of task k's, then task k + 1's.
// A slot is refilled only after the unit it held was consumed: every lane's loads of it
// have landed in registers (an instruction has read them) before the warp got here.
__device__ __forceinline__ void in_top_up(InFeed& F, const NsParams& P, int lane) {
  while (F.issued - F.used < static_cast<uint32_t>(IN_SLOTS)) {
    if (F.cur_iss < F.cur.units()) {
      in_issue(F, F.cur, F.cur_iss++, lane);
      continue;
    }
    if (!F.nxt_known) {
      const uint32_t k1 = F.k + 1;
      // every lane acquires the record's publication itself before reading it
      const bool ready =
          __all_sync(0xffffffffu, mbar_test_cluster(&F.slot_full[k1 % TASK_SLOTS], (k1 / TASK_SLOTS) & 1));
      if (!ready) return;
      F.nxt = input_of(P, F.rec[k1 % TASK_SLOTS], F.row_base, F.half);
      F.nxt_iss = 0;
      F.nxt_known = true;
      // the scheduler acquired the task's inputs; order them before this thread's TMA reads
      if (lane == 0) fence_proxy_async_global();
    }
    if (F.nxt_iss >= F.nxt.units()) return;
    in_issue(F, F.nxt, F.nxt_iss++, lane);
  }
}

// Epilogue of one warp: TMEM lanes of quadrant `quad` (tile rows quad*32 .. quad*32 + 31),
// columns [half * nt/2, (half + 1) * nt/2) of the accumulator at `tacc`, taken as
// 32x32 chunks of two 16-row halves.
// Each 32x32 chunk is staged in the warp's shared buffer and written with a
// TMA bulk store; a symmetric phase also stores the transposed chunk at the
// mirrored position.  A 128-block below the diagonal is not stored at all; in
// a diagonal 128-block the chunks below the diagonal are not stored (their
// mirror covers them) and the chunk on the diagonal is made symmetric before
// its store, so every element is written exactly once.
// The input (A for POLY, X_1's residual for the second step's APPLY) comes through the warp's
// input ring; false if a wait for it ran out.
// fin (the last step's APPLY with LO = 0 only, a run-time choice, so that the kernel holds no
// more inlined copies of this body than one per phase form): FIN_UPDATE also applies S5 to
// the chunk's elements of the bank in place, each lane its own row of the chunk read back from
// the staged bf16 output (so the update uses v exactly as stored), with the bank and mantissa
// loaded at the chunk's start; FIN_ROWSQ also writes the sums of v^2 of the chunk's 32 rows
// over its 32 columns.
template <int EPI, int LO>
__device__ __forceinline__ bool epilogue(const NsParams& P, const EpiJob& J, uint32_t tacc, int quad, int half,
                                         int lane, uint8_t* ebuf, InFeed& F, const volatile int* abort_flag,
                                         int fin = FIN_NONE) {
  // the input: A in POLY (for b A), X_1's residual in the second step's APPLY (for a X_1)
  constexpr bool has_ein = EPI == EPI_POLY || (EPI == EPI_APPLY && LO == LO_READ);
  uint8_t* bufD = ebuf;          // [32 rows][32 cols] bf16, 64-byte swizzle
  uint8_t* bufT = ebuf + 2048;   // [32 cols][32 rows] bf16, 64-byte swizzle (or the residual)
  const int row0 = J.m0 + quad * 32;
  const int I = J.m0 / BM;
  const int ncols = J.nt >> 1;
  const int cbeg = half * ncols;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
  const float ca = P.ca[J.it], cb = P.cb[J.it], cc = P.cc[J.it];
  // The chunk moves as 8x8 matrices in MMA-fragment order (TMEM loads of 16 lanes,
  // ldmatrix / stmatrix through the 64-byte swizzle).  For row half g (rows 16g..16g+15)
  // and column pair p, matrix i covers rows 16g + 8(i & 1) .. and columns 8(2p + (i >> 1)) ..;
  // this thread addresses row `mrow` (of the half) and column group 2p + `mcol`.
  const int mrow = 8 * ((lane >> 3) & 1) + (lane & 7);
  const int mcol = lane >> 4;
  const uint32_t sD = smem_u32(bufD), sT = smem_u32(bufT);
  const bool fin_update = EPI == EPI_APPLY && LO == 0 && fin == FIN_UPDATE;
  const bool fin_rowsq = EPI == EPI_APPLY && LO == 0 && fin == FIN_ROWSQ;

  for (int c = 0; c < ncols; c += 32) {
    const int col0 = J.n0 + cbeg + c;
    // which stores this chunk makes; boxes starting outside the matrix are skipped
    bool direct = row0 < J.M && col0 < J.N, mirror = false, diag = false;
    if (J.sym) {
      const int Jb = col0 / BM;
      if (Jb < I) {
        direct = false;                         // below the diagonal: block (Jb, I) is stored mirrored
      } else if (Jb > I) {
        mirror = direct;
      } else {
        const int cq = (col0 % BM) / 32;
        if (cq < quad) direct = false;          // below the diagonal: the mirror of (cq, quad) covers it
        else if (cq > quad) mirror = direct;
        else diag = direct;
      }
    }
    const bool lo_out = EPI == EPI_APPLY && LO == LO_WRITE && direct;

    float rs[4];   // FIN_ROWSQ: sums of squares of rows 16g + lane/4 (rs[2g]) and 16g + 8 + lane/4 (rs[2g + 1])

    // this chunk's input, both row halves, taken into registers at the chunk's start so that its
    // slot refills under the chunk's work; register 8g + 4p + i holds matrix i of column pair p
    // of row half g
    uint32_t ex[16];
    if (has_ein) {
      in_top_up(F, P, lane);
      const uint32_t slot = F.used % IN_SLOTS;
      if (!mbar_wait_or_abort(&F.full[slot], (F.used / IN_SLOTS) & 1, abort_flag)) return false;
      const uint32_t in = smem_u32(F.buf + slot * IN_BOX_BYTES);
#pragma unroll
      for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int p = 0; p < 2; ++p) ldmatrix_x4(in + sw64(16 * g + mrow, 2 * p + mcol), ex + 8 * g + 4 * p);
      // the loads have landed in registers (an instruction reads them all) before the warp
      // lets lane 0 overwrite their slot
      uint32_t dep = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) dep ^= ex[i];
      asm volatile("mov.b32 %0, %0;" : "+r"(dep));
      F.used += 1;
      __syncwarp();
      if (lane == 0) fence_proxy_async_smem();
      in_top_up(F, P, lane);
    }
    if (lane == 0) bulk_wait_read_all();        // the previous chunk's stores have read the buffers
    __syncwarp();
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      // rows 16g..16g+15 of the chunk: column group j's pairs sit in registers 4j (upper
      // 8 rows) and 4j + 2 (lower 8 rows), as matrix i = 2(j & 1) + (upper ? 0 : 1) of pair j / 2
      uint32_t acc[16];
      tmem_ld_16x256b_x4(tacc + lane_base + (static_cast<uint32_t>(16 * g) << 16) + static_cast<uint32_t>(cbeg + c),
                         acc);
      tmem_ld_wait();
      uint32_t pk[8], pl[8];   // [4p + i], matrix i of column pair p, as the input registers
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int lo8 = 0; lo8 < 2; ++lo8) {
          const int k = 4 * (j >> 1) + 2 * (j & 1) + lo8;
          const float a0 = __uint_as_float(acc[4 * j + 2 * lo8]), a1 = __uint_as_float(acc[4 * j + 2 * lo8 + 1]);
          float o0, o1;
          if (EPI == EPI_GRAM) {
            o0 = J.alpha * a0;
            o1 = J.alpha * a1;
          } else if (EPI == EPI_POLY) {
            o0 = fmaf(cc, a0, cb * bf16_lo(ex[8 * g + k]));
            o1 = fmaf(cc, a1, cb * bf16_hi(ex[8 * g + k]));
            if (diag) {
              // a I on the diagonal: this thread's elements sit at chunk row 16 g + 8 lo8 + lane / 4
              // and columns 8 j + 2 (lane % 4) and the next (a diagonal chunk starts on the diagonal)
              const int lr = 16 * g + 8 * lo8 + (lane >> 2), lc = 8 * j + 2 * (lane & 3);
              if (lr == lc) o0 += ca;
              if (lr == lc + 1) o1 += ca;
            }
          } else if (LO == LO_READ) {
            o0 = fmaf(ca, bf16_lo(ex[8 * g + k]), a0);   // (beta = 1 after the first step)
            o1 = fmaf(ca, bf16_hi(ex[8 * g + k]), a1);
          } else {
            o0 = J.alpha * a0;
            o1 = J.alpha * a1;
          }
          pk[k] = pack_bf16x2(o0, o1);
          // residual o - bf16(o), row-major in the (otherwise idle) transposed buffer
          if (lo_out) pl[k] = pack_bf16x2(o0 - bf16_lo(pk[k]), o1 - bf16_hi(pk[k]));
        }
      }
      if (fin_rowsq) {
        // registers pk[k] with k even hold this thread's two columns of row 16g + lane/4, odd k of
        // row 16g + 8 + lane/4 (columns 8j + 2 (lane % 4) and the next, j = 2 (k / 4) + (k / 2) % 2):
        // squares of the bf16 values v takes, summed in a fixed order.  Columns past the matrix
        // are left out: there the accumulator holds products with the X buffer's row padding,
        // which no phase writes and no store lets out.
        float su = 0.f, sl = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int cl = col0 + 8 * (2 * (k >> 2) + ((k >> 1) & 1)) + 2 * (lane & 3);
          const float e0 = cl < J.N ? bf16_lo(pk[k]) : 0.f, e1 = cl + 1 < J.N ? bf16_hi(pk[k]) : 0.f;
          if (k & 1) {
            sl = fmaf(e0, e0, sl);
            sl = fmaf(e1, e1, sl);
          } else {
            su = fmaf(e0, e0, su);
            su = fmaf(e1, e1, su);
          }
        }
        rs[2 * g] = su;
        rs[2 * g + 1] = sl;
      }
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        if (direct || diag) stmatrix_x4(sD + sw64(16 * g + mrow, 2 * p + mcol), pk + 4 * p);
        // the transposed matrix (rows 16g + 8(i & 1) .., columns 8j ..) lands at rows 8j ..,
        // columns 16g + 8(i & 1) .. of the transposed chunk
        if (mirror || diag)
          stmatrix_x4_trans(sT + sw64(8 * (2 * p + mcol) + (lane & 7), 2 * g + ((lane >> 3) & 1)), pk + 4 * p);
        if (lo_out) stmatrix_x4(sT + sw64(16 * g + mrow, 2 * p + mcol), pl + 4 * p);
      }
    }
    if (diag) {
      __syncwarp();
      // row `lane` of the symmetric diagonal chunk: own values on and above the
      // diagonal, the transposed (upper) values below it
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 t4 = *reinterpret_cast<const uint4*>(bufT + sw64(lane, j));
        const uint4 d4 = *reinterpret_cast<const uint4*>(bufD + sw64(lane, j));
        const uint32_t tw[4] = {t4.x, t4.y, t4.z, t4.w};
        uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c0 = 8 * j + 2 * q;
          const uint32_t lo = (c0 < lane) ? (tw[q] & 0xFFFFu) : (dw[q] & 0xFFFFu);
          const uint32_t hi = (c0 + 1 < lane) ? (tw[q] >> 16) : (dw[q] >> 16);
          dw[q] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(bufD + sw64(lane, j)) = make_uint4(dw[0], dw[1], dw[2], dw[3]);
      }
    }
    if (fin_rowsq) {
      // the four lanes of a row (lanes 4r .. 4r + 3) add their parts, then lane l takes row l's
      // sum (rows 0-7: upper rows of half 0 from lane 4(l & 7); 8-15 lower; 16-31 likewise for
      // half 1) and the warp stores the chunk's 32 row sums as one contiguous run
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 1);
        rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 2);
      }
      const int src = 4 * (lane & 7);
      const float r0 = __shfl_sync(0xffffffffu, rs[0], src), r1 = __shfl_sync(0xffffffffu, rs[1], src);
      const float r2 = __shfl_sync(0xffffffffu, rs[2], src), r3 = __shfl_sync(0xffffffffu, rs[3], src);
      const int sel = lane >> 3;
      const float mine = sel == 0 ? r0 : sel == 1 ? r1 : sel == 2 ? r2 : r3;
      const NsBank& FB = P.bank[J.bi];
      if (direct && row0 + lane < J.M)
        FB.rowsq[(static_cast<size_t>(J.mat) * FB.nchunk + col0 / 32) * J.M + row0 + lane] = mine;
    }
    if (fin_update) {
      __syncwarp();                              // every lane's part of the chunk is staged
      // this lane's row of the chunk (cols are a multiple of 8, so each 8-column piece lies
      // wholly inside or outside the matrix): the bank and mantissa, then v as staged.  The
      // branch on the abort flag (read after the warp's barrier) also keeps these loads from
      // being scheduled ahead into the arithmetic above, where registers are short.
      const int frow = row0 + lane;
      if (direct && frow < J.M && !*abort_flag) {
        const NsBank& FB = P.bank[J.bi];
        const float decay = FB.dscal ? FB.dscal[DSCAL_DECAY] : FB.decay;
        const float neg_lr = FB.dscal ? FB.dscal[DSCAL_NEG_LR] : FB.neg_lr;
        const size_t foff = (static_cast<size_t>(J.mat) * J.M + frow) * J.N + col0;
        // two halves of 16 columns: each half's loads are issued together, then updated
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint4 wv[2], mv[2];
#pragma unroll
          for (int q = 0; q < 2; ++q)
            if (col0 + 16 * h + 8 * q < J.N) {
              wv[q] = *reinterpret_cast<const uint4*>(FB.w + foff + 16 * h + 8 * q);
              mv[q] = *reinterpret_cast<const uint4*>(FB.mant + foff + 16 * h + 8 * q);
            }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int c8 = 16 * h + 8 * q;
            if (col0 + c8 < J.N) {
              // v as stored: row `lane`, columns c8 .. c8 + 7 of the staged chunk
              const uint4 v8 = *reinterpret_cast<const uint4*>(bufD + sw64(lane, 2 * h + q));
              update_eight(wv[q], mv[q], v8, decay, neg_lr);
              *reinterpret_cast<uint4*>(FB.w + foff + c8) = wv[q];
              *reinterpret_cast<uint4*>(FB.mant + foff + c8) = mv[q];
              if (FB.w_copy) *reinterpret_cast<uint4*>(FB.w_copy + foff + c8) = wv[q];
            }
          }
        }
      }
    }
    const bool store_direct = direct && (!fin_update || P.bank[J.bi].store_v);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && (store_direct || mirror)) {
      if (store_direct) tma_store_3d(J.st, bufD, col0, row0, J.mat);
      if (mirror) tma_store_3d(J.st, bufT, row0, col0, J.mat);
      if (lo_out) tma_store_3d(J.st_lo, bufT, col0, row0, J.mat);
      bulk_commit();
    }
  }
  return true;
}

// ---------------------------------------------------------------- kernel

template <bool FIN>
__global__ void __launch_bounds__(GEMM_THREADS, 1) ns_fused_kernel(const __grid_constant__ NsParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_TILE_BYTES;
  uint8_t* sEpi = smem + TILE_SMEM;
  uint8_t* sIn = sEpi + EPI_SMEM;
  uint64_t* full = reinterpret_cast<uint64_t*>(sIn + IN_SMEM);  // [STAGES] (even) both halves landed
  uint64_t* empty = full + STAGES;                // [STAGES] the pair's MMAs are done with the stage
  uint64_t* tfull = empty + STAGES;               // [2] accumulator ready for the epilogue
  uint64_t* tempty = tfull + 2;                   // [2] (even) both CTAs' epilogues drained the accumulator
  uint64_t* slot_full = tempty + 2;               // [TASK_SLOTS] task record written
  uint64_t* slot_empty = slot_full + TASK_SLOTS;  // [TASK_SLOTS] (even) every reader of both CTAs has it
  uint64_t* prod_took = slot_empty + TASK_SLOTS;  // [TASK_SLOTS] (even) the even producer has started the task
  uint64_t* tile_done = prod_took + TASK_SLOTS;   // every epilogue warp's stores of a task are complete
  uint64_t* in_full = tile_done + 2;              // [EPI_WARPS][IN_SLOTS] epilogue input chunk landed
  Task* rec = reinterpret_cast<Task*>(in_full + EPI_WARPS * IN_SLOTS);   // [TASK_SLOTS] (16-byte aligned)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rec + TASK_SLOTS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * EPI_WARPS);
    }
    for (int s = 0; s < TASK_SLOTS; ++s) {
      mbar_init(&slot_full[s], 1);
      mbar_init(&slot_empty[s], even ? SLOT_READERS_EVEN : SLOT_READERS_ODD);
      mbar_init(&prod_took[s], 1);
    }
    mbar_init(tile_done, EPI_WARPS);
    for (int i = 0; i < EPI_WARPS * IN_SLOTS; ++i) mbar_init(&in_full[i], 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();      // both CTAs' barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    latch_status(P.status, DEV_TIMEOUT);
    *abort_flag = 1;
  };
  // The pair's MMAs write the odd CTA's accumulators at the even CTA's TMEM address.
  if (threadIdx.x == 0 && ld_cluster_u32(map_to_rank(tmem_slot, rank ^ 1u)) != tmem) {
    latch_status(P.status, DEV_PAIR_TMEM);
    *abort_flag = 1;
  }
  // A reader of record s reports that it has the task (the odd CTA's relay forwards its
  // CTA's reports to the even CTA's scheduler).
  auto release_slot = [&](int s) { mbar_arrive(&slot_empty[s]); };
  // Every role reads the next pair task from record k % TASK_SLOTS (t < 0 ends the loop).
  auto read_slot = [&](uint32_t k, Task& tk) -> bool {
    const int s = k % TASK_SLOTS;
    if (!mbar_wait_cluster_or_abort(&slot_full[s], (k / TASK_SLOTS) & 1, abort_flag)) {
      fail();
      return false;
    }
    tk = rec[s];
    return true;
  };

  if (warp == SCHED_WARP) {
    if (even && lane == 0) {
      // ---------------- scheduler: claim, decode, wait for the inputs; at most one task ahead of the producer
      const uint32_t rec_odd = map_to_rank(rec, 1);
      for (uint32_t k = 0;; ++k) {
        const int s = k % TASK_SLOTS;
        if (k >= TASK_SLOTS &&
            !mbar_wait_cluster_or_abort(&slot_empty[s], ((k / TASK_SLOTS) - 1) & 1, abort_flag)) {
          fail();
          break;
        }
        if (k >= 1) {
          const uint32_t p = k - 1;
          if (!mbar_wait_or_abort(&prod_took[p % TASK_SLOTS], (p / TASK_SLOTS) & 1, abort_flag)) {
            fail();
            break;
          }
        }
        int t = *abort_flag ? -1 : static_cast<int>(atomicAdd(P.next_task, 1u));
        if (t >= P.total_tasks) t = -1;
        Task tk;
        tk.t = -1;
        if (t >= 0) {
          decode_task(P, t, tk);
          int dit, dph;
          if (dependency(tk, dit, dph)) {
            const NsBank& B = P.bank[tk.bi];
            const unsigned target = static_cast<unsigned>(phase_tiles(B, dph));
            if (!wait_counter(done_counter(B, tk.mat, dit, dph), target, abort_flag)) {
              fail();
              break;   // the consumers see the abort and stop
            }
          }
        }
        rec[s] = tk;
        const uint4* w = reinterpret_cast<const uint4*>(&tk);
        st_cluster_v4(rec_odd + s * sizeof(Task), w[0]);
        st_cluster_v4(rec_odd + s * sizeof(Task) + 16, w[1]);
        mbar_arrive(&slot_full[s]);
        mbar_arrive_cluster(map_to_rank(&slot_full[s], 1));
        if (tk.t < 0) break;
      }
    } else if (!even && lane == 0) {
      // ---------------- relay: once every reader of record k in this CTA has it, one
      // cluster-scope arrival tells the scheduler that the record may be overwritten
      const uint32_t slot_empty_even = map_to_rank(&slot_empty[0], 0);
      for (uint32_t k = 0;; ++k) {
        const int s = k % TASK_SLOTS;
        if (!mbar_wait_cluster_or_abort(&slot_full[s], (k / TASK_SLOTS) & 1, abort_flag)) {
          fail();
          break;
        }
        const bool last = rec[s].t < 0;
        if (!mbar_wait_or_abort(&slot_empty[s], (k / TASK_SLOTS) & 1, abort_flag)) {
          fail();
          break;
        }
        mbar_arrive_cluster(slot_empty_even + 8u * static_cast<uint32_t>(s));
        if (last) break;
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      for (int b = 0; b < P.nbank; ++b) {
        tma_prefetch_map(&P.bank[b].ak);
        tma_prefetch_map(&P.bank[b].bk);
      }
      const uint32_t full_even = map_to_rank(&full[0], 0);
      int st = 0;
      uint32_t ph = 0;
      uint32_t it = 0;
      for (uint32_t k = 0;; ++k) {
        Task tk;
        if (!read_slot(k, tk)) break;
        if (even) mbar_arrive(&prod_took[k % TASK_SLOTS]);
        release_slot(k % TASK_SLOTS);
        if (tk.t < 0 || *abort_flag) break;
        // the scheduler acquired the inputs of this task; order them before this thread's TMA reads
        fence_proxy_async_global();
        const Operands op = task_operands(P.bank[tk.bi], tk);
        const int KB = (op.K + BK - 1) / BK;
        const int m0 = tk.m0 + static_cast<int>(rank) * BM;         // this CTA's A rows
        const int nb0 = tk.n0 + static_cast<int>(rank) * (tk.nt >> 1);   // this CTA's B rows
        const bool load_b = !b_is_a(tk);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          if (it >= STAGES && !mbar_wait_cluster_or_abort(&empty[st], ph ^ 1u, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (even) mbar_expect_tx(&full[st], load_b ? 2u * STAGE_BYTES : 2u * A_TILE_BYTES);   // both CTAs' boxes
          const uint32_t fb = full_even + 8u * static_cast<uint32_t>(st);
          uint8_t* a = sA + st * A_TILE_BYTES;
          uint8_t* b = sB + st * BH_TILE_BYTES;
          const int k0 = kb * BK;
          if (!op.a_mn) tma_load_3d_pair(a, op.a, fb, k0, m0, tk.mat);
          else tma_load_4d_pair(a, op.a, fb, 0, k0, m0 >> 6, tk.mat);
          if (load_b) {
            if (!op.b_mn) tma_load_3d_pair(b, op.b, fb, k0, nb0, tk.mat);
            else tma_load_4d_pair(b, op.b, fb, 0, k0, nb0 >> 6, tk.mat);
          }
          if (++st == STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
      // this CTA stays until the multicast releases of every stage it filled have arrived
      for (uint32_t i = it > STAGES ? it - STAGES : 0u; i < it; ++i) {
        if (!mbar_wait_cluster_or_abort(&empty[i % STAGES], (i / STAGES) & 1, abort_flag)) {
          fail();
          break;
        }
      }
    }
  } else if (warp == 1) {
    if (even && lane == 0) {
      // ---------------- MMA issuer of the pair
      uint32_t it = 0;
      for (uint32_t k = 0;; ++k) {
        Task tk;
        if (!read_slot(k, tk)) break;
        release_slot(k % TASK_SLOTS);
        if (tk.t < 0 || *abort_flag) break;
        const Operands op = task_operands(P.bank[tk.bi], tk);
        const int KB = (op.K + BK - 1) / BK;
        const uint32_t buf = k & 1;
        if (k >= 2 && !mbar_wait_cluster_or_abort(&tempty[buf], ((k >> 1) - 1) & 1, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t dacc = tmem + buf * ACC_COLS;
        const uint32_t idesc = idesc_bf16_m256(tk.nt, op.a_mn, op.b_mn);
        const uint32_t a_step = op.a_mn ? 2048u : 32u, b_step = op.b_mn ? 2048u : 32u;
        const uint32_t a_lbo = op.a_mn ? 8192u : 16u, b_lbo = op.b_mn ? 8192u : 16u;
        const bool b_from_a = b_is_a(tk);   // then a_mn == b_mn: the same steps and strides
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = it % STAGES;
          if (!mbar_wait_or_abort(&full[st], (it / STAGES) & 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + st * A_TILE_BYTES);
          const uint32_t b0 = b_from_a ? a0 : smem_u32(sB + st * BH_TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            umma_bf16_pair(dacc, smem_desc_sw128(a0 + kk * a_step, a_lbo, 1024),
                           smem_desc_sw128(b0 + kk * b_step, b_lbo, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair_both(&empty[st]);   // the stage may be refilled in both CTAs
        }
        umma_commit_pair_both(&tfull[buf]);
        if (!ok) break;
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* ebuf = sEpi + (warp - 2) * EPI_BUF_BYTES;
    const uint32_t tempty_even = map_to_rank(&tempty[0], 0);
    InFeed F;
    F.buf = sIn + (warp - 2) * IN_SLOTS * IN_BOX_BYTES;
    F.full = in_full + (warp - 2) * IN_SLOTS;
    F.rec = rec;
    F.slot_full = slot_full;
    F.issued = F.used = 0;
    F.cur_iss = F.nxt_iss = 0;
    F.cur.nch = F.nxt.nch = 0;
    F.nxt_known = false;
    F.row_base = static_cast<int>(rank) * BM + quad * 32;
    F.half = half;
    for (uint32_t k = 0;; ++k) {
      Task tk;
      if (!read_slot(k, tk)) break;
      // the input of task k: already known (and partly issued) if the ring ran ahead into it
      F.k = k;
      if (F.nxt_known) {
        F.cur = F.nxt;
        F.cur_iss = F.nxt_iss;
        F.nxt_known = false;
      } else {
        F.cur = input_of(P, tk, F.row_base, half);
        F.cur_iss = 0;
        if (lane == 0) fence_proxy_async_global();
      }
      __syncwarp();
      if (lane == 0) release_slot(k % TASK_SLOTS);
      if (tk.t < 0) break;
      in_top_up(F, P, lane);                     // this task's first input chunks, under its MMAs
      const NsBank& B = P.bank[tk.bi];
      const uint32_t buf = k & 1;
      if (!mbar_wait_or_abort(&tfull[buf], (k >> 1) & 1, abort_flag)) {
        fail();
        break;
      }
      if (*abort_flag) break;
      tc_fence_after();
      EpiJob J;
      J.mat = tk.mat;
      J.it = tk.it;
      J.m0 = tk.m0 + static_cast<int>(rank) * BM;   // this CTA's rows of the pair tile
      J.n0 = tk.n0;
      J.nt = tk.nt;
      J.alpha = 1.f;
      J.st_lo = nullptr;
      J.bi = tk.bi;
      const uint32_t tacc = tmem + buf * ACC_COLS;
      bool ok;
      if (tk.ph == EPI_GRAM) {
        if (tk.it == 0) {
          const float sc = B.scale[tk.mat];
          J.alpha = sc * sc;
        }
        J.st = &B.st_a;
        J.M = J.N = B.m;
        J.sym = 1;
        ok = epilogue<EPI_GRAM, 0>(P, J, tacc, quad, half, lane, ebuf, F, abort_flag);
      } else if (tk.ph == EPI_POLY) {
        J.st = &B.st_b;
        J.M = J.N = B.m;
        J.sym = 1;
        ok = epilogue<EPI_POLY, 0>(P, J, tacc, quad, half, lane, ebuf, F, abort_flag);
      } else {
        if (tk.it == 0) J.alpha = B.scale[tk.mat];
        J.st = &B.st_x[iterate_buffer(tk.it + 1)];
        // X_1's residual waits in x[2], which the second APPLY overwrites tile by tile only
        // after each chunk has read its own part (through the input ring, as input_of sets up
        // for step 1)
        if (tk.it == 0 && P.steps > 1) J.st_lo = &B.st_x[2];
        J.M = B.tall ? B.n : B.m;
        J.N = B.tall ? B.m : B.n;
        J.sym = 0;
        // only the FIN instantiation carries the last-step modes (the plain kernel holds none of
        // their code); the host asks for one only with at least 3 steps, so the last step's APPLY
        // neither writes nor reads X_1's residual
        const int fin = (FIN && tk.it == P.steps - 1) ? B.fin : FIN_NONE;
        if (J.st_lo)
          ok = epilogue<EPI_APPLY, LO_WRITE>(P, J, tacc, quad, half, lane, ebuf, F, abort_flag);
        else if (tk.it == 1)
          ok = epilogue<EPI_APPLY, LO_READ>(P, J, tacc, quad, half, lane, ebuf, F, abort_flag);
        else
          ok = epilogue<EPI_APPLY, 0>(P, J, tacc, quad, half, lane, ebuf, F, abort_flag, fin);
      }
      if (!ok) {
        fail();
        break;
      }
      in_top_up(F, P, lane);                     // the next task's first chunks, under this one's store waits
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_remote(tempty_even + 8u * buf);    // the even CTA's MMA issuer may reuse the accumulator
        bulk_wait_all();                         // this warp's part of the tile is in global memory
        mbar_arrive(tile_done);
      }
      // one thread publishes the tile once every epilogue warp's stores are complete; it
      // observes completion k before its own arrival for task k+1, so no phase is skipped
      if (warp == 2 && lane == 0) {
        if (mbar_wait_or_abort(tile_done, k & 1, abort_flag)) {
          fence_proxy_async_global();
          red_release_add(done_counter(B, tk.mat, tk.it, tk.ph), 1u);
        } else {
          fail();
        }
      }
      __syncwarp();
    }
    // input chunks still in flight (only after an abort) land before the CTA exits
    for (; F.used != F.issued; ++F.used)
      if (!mbar_wait(&F.full[F.used % IN_SLOTS], (F.used / IN_SLOTS) & 1)) break;
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();      // no multicast or remote arrival targets a CTA that has left
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// The launch of one instantiation: per-device set-up (shared-memory opt-in, the number of
// co-resident CTA pairs) is done by the first call on each device; concurrent first calls from
// several host threads do the same idempotent work.
template <bool FIN>
cudaError_t launch_ns_kernel(const NsParams& p, cudaStream_t s) {
  static std::atomic<bool> attr_done[64];
  static std::atomic<int> max_clusters[64];
  if (p.total_tasks == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(ns_fused_kernel<FIN>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = GEMM_SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int npairs = max_clusters[dev].load(std::memory_order_relaxed);
  if (npairs == 0) {
    // one pair per two SMs, as many as can be resident at once (every pair must be)
    cfg.gridDim = dim3(2, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&npairs, reinterpret_cast<const void*>(ns_fused_kernel<FIN>), &cfg);
    if (e != cudaSuccess) return e;
    if (npairs <= 0) return cudaErrorInvalidConfiguration;
    max_clusters[dev].store(npairs, std::memory_order_relaxed);
  }
  const int pairs = p.total_tasks < npairs ? p.total_tasks : npairs;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  e = cudaLaunchKernelEx(&cfg, ns_fused_kernel<FIN>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace
}  // namespace mb
