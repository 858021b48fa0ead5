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
// CTA = 6 warps, one output tile of 128 x (128|256) fp32 in TMEM:
//   warp 0 lane 0 : TMA producer, STAGES-deep ring of (A 128x64, B 256x64) bf16 tiles
//   warp 1        : TMEM allocation; lane 0 issues tcgen05.mma (K = 16 per instruction)
//   warps 2..5    : epilogue, tcgen05.ld of their 32 TMEM lanes, fp32 math, bf16 stores
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
constexpr int GEMM_SMEM = TILE_SMEM + 1024 /* alignment slack */ + 256 /* barriers */;
constexpr int GEMM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;

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

// 32 consecutive bf16 of one row -> fp32 (zeros outside [0, ncols) or a masked row).
__device__ __forceinline__ void load_row32(const uint16_t* base, long long ld, int row, int col0, int ncols,
                                           bool row_ok, float (&v)[32]) {
  if (row_ok && col0 + 32 <= ncols) {
    const uint4* p = reinterpret_cast<const uint4*>(base + static_cast<long long>(row) * ld + col0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 w = p[j];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * j + 2 * i] = bf16_bits_to_float(ws[i] & 0xFFFFu);
        v[8 * j + 2 * i + 1] = bf16_bits_to_float(ws[i] >> 16);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      v[i] = (row_ok && col0 + i < ncols) ? bf16_bits_to_float(base[static_cast<long long>(row) * ld + col0 + i])
                                          : 0.f;
  }
}

__device__ __forceinline__ void store_row32(uint16_t* base, long long ld, int row, int col0, int ncols,
                                            bool row_ok, const float (&o)[32]) {
  if (!row_ok) return;
  if (col0 + 32 <= ncols) {
    uint4* p = reinterpret_cast<uint4*>(base + static_cast<long long>(row) * ld + col0);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      p[j] = make_uint4(pack_bf16x2(o[8 * j + 0], o[8 * j + 1]), pack_bf16x2(o[8 * j + 2], o[8 * j + 3]),
                        pack_bf16x2(o[8 * j + 4], o[8 * j + 5]), pack_bf16x2(o[8 * j + 6], o[8 * j + 7]));
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i < ncols)
        base[static_cast<long long>(row) * ld + col0 + i] = static_cast<uint16_t>(float_to_bf16_bits(o[i]));
  }
}

template <int EPI>
__device__ __forceinline__ void epilogue(const GemmParams& P, const GemmProblem& pr, const Tile& tl,
                                         uint32_t tmem, int quad, int lane) {
  const int row = tl.m0 + quad * 32 + lane;
  const bool row_ok = row < pr.M;
  float alpha = 1.f;
  if (pr.scale) {
    const float s = pr.scale[tl.mat];
    alpha = (EPI == EPI_GRAM) ? s * s : s;
  }
  uint16_t* out = pr.out + tl.mat * pr.out_ms;
  const uint16_t* ein = (EPI == EPI_GRAM) ? nullptr : pr.ein + tl.mat * pr.ein_ms;
  const int I = tl.m0 / BM;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

  for (int c0 = 0; c0 < tl.nt; c0 += 32) {
    uint32_t acc[32];
    tmem_ld_32x32(tmem + lane_base + static_cast<uint32_t>(c0), acc);
    tmem_ld_wait();
    const int col0 = tl.n0 + c0;
    float o[32];
    if (EPI == EPI_GRAM) {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = alpha * __uint_as_float(acc[i]);
    } else {
      float e[32];
      load_row32(ein, pr.ein_ld, row, col0, pr.N, row_ok, e);
      if (EPI == EPI_POLY) {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = fmaf(P.cc, __uint_as_float(acc[i]), P.cb * e[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = alpha * fmaf(P.ca, e[i], __uint_as_float(acc[i]));
      }
    }
    if (pr.sym) {
      const int J = col0 / BM;
      if (J == I) {
        // diagonal block: the upper half (with the diagonal) directly, the strict upper mirrored
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int col = col0 + i;
          if (!row_ok || col >= pr.N) continue;
          const uint16_t b = static_cast<uint16_t>(float_to_bf16_bits(o[i]));
          if (col >= row) out[static_cast<long long>(row) * pr.out_ld + col] = b;
          if (col > row) out[static_cast<long long>(col) * pr.out_ld + row] = b;
        }
      } else {
        store_row32(out, pr.out_ld, row, col0, pr.N, row_ok, o);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int col = col0 + i;
            if (col < pr.N)
              out[static_cast<long long>(col) * pr.out_ld + row] = static_cast<uint16_t>(float_to_bf16_bits(o[i]));
          }
        }
      }
    } else {
      store_row32(out, pr.out_ld, row, col0, pr.N, row_ok, o);
    }
  }
}

template <int EPI>
__global__ void __launch_bounds__(GEMM_THREADS, 1) ns_gemm_kernel(const __grid_constant__ GemmParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_TILE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + TILE_SMEM);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Tile tl;
  const bool valid = decode_tile(P, blockIdx.x, tl);
  const GemmProblem& pr = P.prob[valid ? tl.pi : 0];

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
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

  if (valid) {
    const int KB = (pr.K + BK - 1) / BK;
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_map(&pr.map_a);
      tma_prefetch_map(&pr.map_b);
      const uint32_t bytes = A_TILE_BYTES + tl.nt * BK * 2;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % STAGES;
        if (kb >= STAGES && !mbar_wait(&empty[s], ((kb / STAGES) - 1) & 1)) {
          latch_status(P.status, DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
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
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc = idesc_bf16_m128(tl.nt, pr.a_mn, pr.b_mn);
      const uint32_t a_step = pr.a_mn ? 2048u : 32u, b_step = pr.b_mn ? 2048u : 32u;
      const uint32_t a_lbo = pr.a_mn ? 8192u : 16u, b_lbo = pr.b_mn ? 8192u : 16u;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(&full[s], (kb / STAGES) & 1)) {
          latch_status(P.status, DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + s * A_TILE_BYTES), b0 = smem_u32(sB + s * B_TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          umma_bf16(tmem, smem_desc_sw128(a0 + kk * a_step, a_lbo, 1024),
                    smem_desc_sw128(b0 + kk * b_step, b_lbo, 1024), idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      umma_commit(accf);
    } else if (warp >= 2) {
      // ---------------- epilogue
      if (!mbar_wait(accf, 0)) {
        latch_status(P.status, DEV_TIMEOUT);
      } else if (!*abort_flag) {
        tc_fence_after();
        epilogue<EPI>(P, pr, tl, tmem, warp & 3, lane);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

bool g_attr_done[3][64];

}  // namespace

cudaError_t launch_gemm(const GemmParams& p, int epi, cudaStream_t s) {
  if (p.total_tiles == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const void* fn = nullptr;
  switch (epi) {
    case EPI_GRAM: fn = reinterpret_cast<const void*>(ns_gemm_kernel<EPI_GRAM>); break;
    case EPI_POLY: fn = reinterpret_cast<const void*>(ns_gemm_kernel<EPI_POLY>); break;
    default: fn = reinterpret_cast<const void*>(ns_gemm_kernel<EPI_APPLY>); break;
  }
  const int ei = (epi == EPI_GRAM) ? 0 : (epi == EPI_POLY) ? 1 : 2;
  if (dev < 64 && !g_attr_done[ei][dev]) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
    if (e != cudaSuccess) return e;
    g_attr_done[ei][dev] = true;
  }
  switch (epi) {
    case EPI_GRAM: ns_gemm_kernel<EPI_GRAM><<<p.total_tiles, GEMM_THREADS, GEMM_SMEM, s>>>(p); break;
    case EPI_POLY: ns_gemm_kernel<EPI_POLY><<<p.total_tiles, GEMM_THREADS, GEMM_SMEM, s>>>(p); break;
    default: ns_gemm_kernel<EPI_APPLY><<<p.total_tiles, GEMM_THREADS, GEMM_SMEM, s>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace mb
