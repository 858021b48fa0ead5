// Batched Newton-Schulz GEMMs on the sm_103a tensor cores (tcgen05 + TMEM,
// operands staged by TMA with 128-byte swizzle).
//
// One quintic step ("Muon Custom Sizing" write-up, section 2.3; Track-2
// record 7 write-up, section 4.2) is three GEMM phases over every matrix of
// the bank(s) in the launch:
//   EPI_GRAM   A  = alpha * X X^T       (alpha = s^2 on the first step, s = 1/(||u||+eps))
//   EPI_POLY   B  = b A + c A A         (A symmetric, so A A = A A^T)
//   EPI_APPLY  X' = beta (a X + B X)    (beta = s on the first step)
// A tall slice (rows > cols) stays in its stored orientation and runs the
// swapped-operand form A = X^T X, X' = beta (a X + X B); the difference is
// only which operand tiles are K-major and which are MN-major.
//
// A and B are symmetric: those phases compute only the 128x128 blocks on or
// above the diagonal (paired into 128x256 tiles) and store each off-diagonal
// block twice, directly and mirrored, so the next phase reads a full matrix.
//
// Persistent CTAs, one per SM, take output tiles of 128 x (128|256) round-robin.
//   warp 0 lane 0 : TMA producer, STAGES-deep ring of (A 128x64, B 256x64) bf16 tiles
//   warp 1        : owns 512 TMEM columns = two 256-column fp32 accumulators;
//                   lane 0 issues tcgen05.mma (K = 16 per instruction)
//   warps 2..9    : epilogue, two warps per 32-lane TMEM quadrant (each takes half
//                   the columns); tile t's epilogue runs under tile t+1's MMAs
#include "mb_device.cuh"
#include "mb_internal.h"

namespace mb {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_TILE_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_TILE_BYTES = 256 * BK * 2;  // 32 KB
constexpr int TILE_SMEM = STAGES * (A_TILE_BYTES + B_TILE_BYTES);
constexpr int EPI_WARPS = 8;
constexpr int EPI_BUF_BYTES = 4096;          // per epilogue warp: 32x32 bf16 chunk + its transpose
constexpr int EPI_SMEM = EPI_WARPS * EPI_BUF_BYTES;
constexpr int GEMM_SMEM = TILE_SMEM + EPI_SMEM + 1024 /* alignment slack */ + 256 /* barriers */;
constexpr int GEMM_THREADS = 32 * (2 + EPI_WARPS);
constexpr uint32_t ACC_COLS = 256;          // one accumulator
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;

struct Tile {
  int pi, mat, m0, n0, nt;
};

__device__ __forceinline__ bool decode_tile(const GemmParams& P, int t, Tile& tl) {
  for (int pi = 0; pi < P.nprob; ++pi) {
    const GemmProblem& pr = P.prob[pi];
    const int cnt = pr.batch * pr.tiles_per_mat;
    if (t >= pr.tile_begin + cnt) continue;
    int lt = t - pr.tile_begin;
    tl.pi = pi;
    tl.mat = lt / pr.tiles_per_mat;
    lt -= tl.mat * pr.tiles_per_mat;
    if (pr.sym) {
      for (int I = 0; I < pr.T; ++I) {
        const int c = (pr.T - I + 1) >> 1;
        if (lt < c) {
          const int J = I + 2 * lt;
          tl.m0 = I * BM;
          tl.n0 = J * BM;
          tl.nt = (J + 1 < pr.T) ? 256 : 128;
          return true;
        }
        lt -= c;
      }
      return false;
    }
    const int tm = lt / pr.tn, tj = lt - tm * pr.tn;
    tl.m0 = tm * BM;
    tl.n0 = tj * 256;
    tl.nt = (pr.N - tl.n0 > 128) ? 256 : 128;
    return true;
  }
  return false;
}

// 32 consecutive bf16 of one row as 16 packed words (zeros outside [0, ncols) or a masked row).
__device__ __forceinline__ void load_row32_raw(const uint16_t* base, long long ld, int row, int col0, int ncols,
                                               bool row_ok, uint32_t (&w)[16]) {
  if (row_ok && col0 + 32 <= ncols) {
    const uint4* p = reinterpret_cast<const uint4*>(base + static_cast<long long>(row) * ld + col0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = p[j];
      w[4 * j + 0] = v.x;
      w[4 * j + 1] = v.y;
      w[4 * j + 2] = v.z;
      w[4 * j + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t lo = 0, hi = 0;
      if (row_ok && col0 + 2 * i < ncols) lo = base[static_cast<long long>(row) * ld + col0 + 2 * i];
      if (row_ok && col0 + 2 * i + 1 < ncols) hi = base[static_cast<long long>(row) * ld + col0 + 2 * i + 1];
      w[i] = lo | (hi << 16);
    }
  }
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a [32][32] bf16 staging
// buffer laid out as the TMA 64-byte swizzle expects (address bits [4,6) XOR
// bits [7,9)): row-wise 16-byte writes of a warp then hit distinct banks.
__device__ __forceinline__ uint32_t sw64(int row, int chunk) {
  return static_cast<uint32_t>(row * 64 + 16 * (chunk ^ ((row >> 1) & 3)));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return bf16_bits_to_float(w & 0xFFFFu); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return bf16_bits_to_float(w >> 16); }

// Epilogue of one warp: TMEM lanes of quadrant `quad` (tile rows quad*32 + lane),
// columns [half * nt/2, (half + 1) * nt/2) of the accumulator at `tacc`.
// Each 32x32 chunk is staged in the warp's shared buffer and written with a
// TMA bulk store; a symmetric phase also stores the transposed chunk at the
// mirrored position.  In a diagonal 128-block the chunks below the diagonal
// are not stored (their mirror covers them) and the chunk on the diagonal is
// made symmetric before its store, so every element is written exactly once.
template <int EPI>
__device__ __forceinline__ void epilogue(const GemmParams& P, const GemmProblem& pr, const Tile& tl,
                                         uint32_t tacc, int quad, int half, int lane, uint8_t* ebuf) {
  uint8_t* bufD = ebuf;          // [32 rows][32 cols] bf16, 64-byte swizzle
  uint8_t* bufT = ebuf + 2048;   // [32 cols][32 rows] bf16, 64-byte swizzle
  const int row0 = tl.m0 + quad * 32;
  const int row = row0 + lane;
  const bool row_ok = row < pr.M;
  float alpha = 1.f;
  if (pr.scale) {
    const float s = pr.scale[tl.mat];
    alpha = (EPI == EPI_GRAM) ? s * s : s;
  }
  const uint16_t* ein = (EPI == EPI_GRAM) ? nullptr : pr.ein + tl.mat * pr.ein_ms;
  const int I = tl.m0 / BM;
  const int ncols = tl.nt >> 1;
  const int cbeg = half * ncols;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

  uint32_t e_cur[16], e_nxt[16];
  if (EPI != EPI_GRAM) load_row32_raw(ein, pr.ein_ld, row, tl.n0 + cbeg, pr.N, row_ok, e_cur);

  for (int c = 0; c < ncols; c += 32) {
    const int col0 = tl.n0 + cbeg + c;
    if (EPI != EPI_GRAM && c + 32 < ncols) load_row32_raw(ein, pr.ein_ld, row, col0 + 32, pr.N, row_ok, e_nxt);
    uint32_t acc[32];
    tmem_ld_32x32(tacc + lane_base + static_cast<uint32_t>(cbeg + c), acc);
    tmem_ld_wait();
    float o[32];
    if (EPI == EPI_GRAM) {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = alpha * __uint_as_float(acc[i]);
    } else if (EPI == EPI_POLY) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[2 * i] = fmaf(P.cc, __uint_as_float(acc[2 * i]), P.cb * bf16_lo(e_cur[i]));
        o[2 * i + 1] = fmaf(P.cc, __uint_as_float(acc[2 * i + 1]), P.cb * bf16_hi(e_cur[i]));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[2 * i] = alpha * fmaf(P.ca, bf16_lo(e_cur[i]), __uint_as_float(acc[2 * i]));
        o[2 * i + 1] = alpha * fmaf(P.ca, bf16_hi(e_cur[i]), __uint_as_float(acc[2 * i + 1]));
      }
    }
    if (EPI != EPI_GRAM) {
#pragma unroll
      for (int i = 0; i < 16; ++i) e_cur[i] = e_nxt[i];
    }

    // which stores this chunk makes; boxes starting outside the matrix are skipped
    bool direct = row0 < pr.M && col0 < pr.N, mirror = false, diag = false;
    if (pr.sym) {
      const int J = col0 / BM;
      if (J != I) {
        mirror = direct;
      } else {
        const int cq = (col0 % BM) / 32;
        if (cq < quad) direct = false;          // below the diagonal: the mirror of (cq, quad) covers it
        else if (cq > quad) mirror = direct;
        else diag = direct;
      }
    }
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);

    if (lane == 0) bulk_wait_read_all();        // the previous chunk's stores have read the buffers
    __syncwarp();
    if (mirror || diag) {
      const uint32_t lane_off = 2u * (lane & 7);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        *reinterpret_cast<uint16_t*>(bufT + sw64(2 * i, lane >> 3) + lane_off) = static_cast<uint16_t>(pk[i] & 0xFFFFu);
        *reinterpret_cast<uint16_t*>(bufT + sw64(2 * i + 1, lane >> 3) + lane_off) = static_cast<uint16_t>(pk[i] >> 16);
      }
    }
    if (diag) {
      __syncwarp();
      // row `lane` of the symmetric diagonal chunk: own values on and above the
      // diagonal, the transposed (upper) values below it
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 t4 = *reinterpret_cast<const uint4*>(bufT + sw64(lane, j));
        const uint32_t tw[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c0 = 8 * j + 2 * k;
          const uint32_t lo = (c0 < lane) ? (tw[k] & 0xFFFFu) : (pk[4 * j + k] & 0xFFFFu);
          const uint32_t hi = (c0 + 1 < lane) ? (tw[k] >> 16) : (pk[4 * j + k] >> 16);
          pk[4 * j + k] = lo | (hi << 16);
        }
      }
    }
    if (direct) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(bufD + sw64(lane, j)) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && (direct || mirror)) {
      if (direct) tma_store_3d(&pr.map_out, bufD, col0, row0, tl.mat);
      if (mirror) tma_store_3d(&pr.map_out, bufT, row0, col0, tl.mat);
      bulk_commit();
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1) ns_gemm_kernel(const __grid_constant__ GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_TILE_BYTES;
  uint8_t* sEpi = smem + TILE_SMEM;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TILE_SMEM + EPI_SMEM);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;    // [2] accumulator ready for the epilogue
  uint64_t* tempty = tfull + 2;        // [2] accumulator drained by the epilogue
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int first = blockIdx.x, stride = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], EPI_WARPS);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    latch_status(P.status, DEV_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      for (int pi = 0; pi < P.nprob; ++pi) {
        tma_prefetch_map(&P.prob[pi].map_a);
        tma_prefetch_map(&P.prob[pi].map_b);
      }
      uint32_t it = 0;
      for (int t = first; t < P.total_tiles && !*abort_flag; t += stride) {
        Tile tl;
        if (!decode_tile(P, t, tl)) break;
        const GemmProblem& pr = P.prob[tl.pi];
        const int KB = (pr.K + BK - 1) / BK;
        const uint32_t bytes = A_TILE_BYTES + tl.nt * BK * 2;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t use = it / STAGES;
          if (use > 0 && !mbar_wait_or_abort(&empty[s], (use - 1) & 1, abort_flag)) {
            fail();
            break;
          }
          mbar_expect_tx(&full[s], bytes);
          uint8_t* a = sA + s * A_TILE_BYTES;
          uint8_t* b = sB + s * B_TILE_BYTES;
          const int k0 = kb * BK;
          if (!pr.a_mn) {
            tma_load_3d(a, &pr.map_a, &full[s], k0, tl.m0, tl.mat);
          } else {
            tma_load_3d(a, &pr.map_a, &full[s], tl.m0, k0, tl.mat);
            tma_load_3d(a + 8192, &pr.map_a, &full[s], tl.m0 + 64, k0, tl.mat);
          }
          if (!pr.b_mn) {
            for (int h = 0; h < tl.nt / 128; ++h)
              tma_load_3d(b + h * 16384, &pr.map_b, &full[s], k0, tl.n0 + 128 * h, tl.mat);
          } else {
            for (int h = 0; h < tl.nt / 64; ++h)
              tma_load_3d(b + h * 8192, &pr.map_b, &full[s], tl.n0 + 64 * h, k0, tl.mat);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      uint32_t it = 0, j = 0;
      for (int t = first; t < P.total_tiles && !*abort_flag; t += stride, ++j) {
        Tile tl;
        if (!decode_tile(P, t, tl)) break;
        const GemmProblem& pr = P.prob[tl.pi];
        const int KB = (pr.K + BK - 1) / BK;
        const uint32_t buf = j & 1;
        if (j >= 2 && !mbar_wait_or_abort(&tempty[buf], ((j >> 1) - 1) & 1, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t dacc = tmem + buf * ACC_COLS;
        const uint32_t idesc = idesc_bf16_m128(tl.nt, pr.a_mn, pr.b_mn);
        const uint32_t a_step = pr.a_mn ? 2048u : 32u, b_step = pr.b_mn ? 2048u : 32u;
        const uint32_t a_lbo = pr.a_mn ? 8192u : 16u, b_lbo = pr.b_mn ? 8192u : 16u;
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait_or_abort(&full[s], (it / STAGES) & 1, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * A_TILE_BYTES), b0 = smem_u32(sB + s * B_TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            umma_bf16(dacc, smem_desc_sw128(a0 + kk * a_step, a_lbo, 1024),
                      smem_desc_sw128(b0 + kk * b_step, b_lbo, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        umma_commit(&tfull[buf]);
        if (!ok) break;
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    uint32_t j = 0;
    for (int t = first; t < P.total_tiles; t += stride, ++j) {
      Tile tl;
      if (!decode_tile(P, t, tl)) break;
      const uint32_t buf = j & 1;
      if (!mbar_wait_or_abort(&tfull[buf], (j >> 1) & 1, abort_flag)) {
        fail();
        break;
      }
      if (*abort_flag) break;
      tc_fence_after();
      epilogue<EPI>(P, P.prob[tl.pi], tl, tmem + buf * ACC_COLS, quad, half, lane,
                    sEpi + (warp - 2) * EPI_BUF_BYTES);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
    }
    if (lane == 0) bulk_wait_all();              // this warp's bulk stores are complete
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

bool g_attr_done[3][64];
int g_num_sms[64];

}  // namespace

cudaError_t launch_gemm(const GemmParams& p, int epi, cudaStream_t s) {
  if (p.total_tiles == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const void* fn = nullptr;
  switch (epi) {
    case EPI_GRAM: fn = reinterpret_cast<const void*>(ns_gemm_kernel<EPI_GRAM>); break;
    case EPI_POLY: fn = reinterpret_cast<const void*>(ns_gemm_kernel<EPI_POLY>); break;
    default: fn = reinterpret_cast<const void*>(ns_gemm_kernel<EPI_APPLY>); break;
  }
  const int ei = (epi == EPI_GRAM) ? 0 : (epi == EPI_POLY) ? 1 : 2;
  if (!g_attr_done[ei][dev]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (e != cudaSuccess) return e;
    g_attr_done[ei][dev] = true;
  }
  if (g_num_sms[dev] == 0) {
    e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const int grid = p.total_tiles < g_num_sms[dev] ? p.total_tiles : g_num_sms[dev];
  switch (epi) {
    case EPI_GRAM: ns_gemm_kernel<EPI_GRAM><<<grid, GEMM_THREADS, GEMM_SMEM, s>>>(p); break;
    case EPI_POLY: ns_gemm_kernel<EPI_POLY><<<grid, GEMM_THREADS, GEMM_SMEM, s>>>(p); break;
    default: ns_gemm_kernel<EPI_APPLY><<<grid, GEMM_THREADS, GEMM_SMEM, s>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace mb
