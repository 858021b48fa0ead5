// Bandwidth-bound stages of the Muon bank step and the small-matrix
// Newton-Schulz path.
//
//   k1_kernel      S1 momentum (lerp form, "Muon Custom Sizing" write-up,
//                  section 4) writing u in bf16, plus per-chunk sums of u^2
//                  for the Frobenius normalisation (S2).  128-bit loads and
//                  stores, warp-shuffle reductions in a fixed order; the
//                  arithmetic is the warp units of mb_ew_units.cuh.
//   scale_kernel   s = 1/(||u||_F + 1e-7) per matrix from those partial sums.
//   small_ns       the quintic iteration (same write-up, section 2.3) in fp32
//                  for matrices with min(rows, cols) <= 64.
//   row_sumsq /    NorMuon reading: per-row sums of v^2, the second-moment
//   row_scale      EMA and the Frobenius-preserving per-row factor.
//   k3_kernel      S5 mixed-precision update (Track-2 record 7 write-up,
//                  section 4.1): fp32 from bf16 + mantissa, decay, scaled
//                  step, truncating split.
#include <atomic>

#include "mb_device.cuh"
#include "mb_ew_units.cuh"
#include "mb_internal.h"

namespace mb {

namespace {

constexpr float NS_EPS = 1e-7f;
constexpr float NORMUON_FLOOR = 1e-10f;

__device__ __forceinline__ int ew_bank(const EwParams& p) {
  int bi = 0;
  while (bi + 1 < p.nb && static_cast<int>(blockIdx.x) >= p.b[bi + 1].block_begin) ++bi;
  return bi;
}

// ---------------------------------------------------------------- S1 (+ S2 partials)

template <bool MOMENTUM>
__global__ void __launch_bounds__(EW_THREADS) k1_kernel(const __grid_constant__ EwParams p) {
  __shared__ float red[EW_UNITS_PER_CHUNK];
  const EwBank& B = p.b[ew_bank(p)];
  const int local = blockIdx.x - B.block_begin;
  const int mat = local / B.P, chunk = local - mat * B.P;
  const int E = B.rows * B.cols;
  const int e0 = chunk * EW_CHUNK;
  const int e1 = min(E, e0 + EW_CHUNK);
  const size_t moff = static_cast<size_t>(mat) * E;
  const float mu = B.dscal ? B.dscal[DSCAL_MU] : p.mu, omm = B.dscal ? B.dscal[DSCAL_OMM] : p.omm;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // each warp is one unit of the chunk; the chunk's sum of u^2 adds the units' in warp order
  const float ss = momentum_unit<MOMENTUM>(B.src + moff, MOMENTUM ? B.mom + moff : nullptr,
                                           B.xout + static_cast<size_t>(mat) * B.rows * B.out_ld, B.cols, B.out_ld,
                                           e0, e1, w, lane, mu, omm);
  if (lane == 0) red[w] = ss;
  __syncthreads();
  if (threadIdx.x == 0 && B.partials) {
    float t = 0.f;
    for (int i = 0; i < EW_UNITS_PER_CHUNK; ++i) t += red[i];
    B.partials[static_cast<size_t>(mat) * B.P + chunk] = t;
  }
}

// ---------------------------------------------------------------- S2 finalise

__global__ void __launch_bounds__(256) scale_kernel(const __grid_constant__ ScaleParams p) {
  const int gm = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gm >= p.total_mats) return;
  int bi = 0;
  while (bi + 1 < p.nb && gm >= p.b[bi + 1].mat_begin) ++bi;
  const ScaleBank& B = p.b[bi];
  const int mat = gm - B.mat_begin;
  const float s = scale_from_units(B.partials + static_cast<size_t>(mat) * B.P, B.P, lane);
  if (lane == 0) B.scale[mat] = s;
}

// ns_steps == 0: v = bf16(s * u)
__global__ void __launch_bounds__(EW_THREADS) ns0_kernel(const __grid_constant__ EwParams p) {
  const EwBank& B = p.b[ew_bank(p)];
  const int local = blockIdx.x - B.block_begin;
  const int mat = local / B.P, chunk = local - mat * B.P;
  const int E = B.rows * B.cols;
  const int e0 = chunk * EW_CHUNK, e1 = min(E, e0 + EW_CHUNK);
  const float s = B.scale[mat];
  const uint16_t* xi = B.xin + static_cast<size_t>(mat) * B.rows * B.ld;
  uint16_t* xo = B.xout + static_cast<size_t>(mat) * B.rows * B.out_ld;
  for (int e = e0 + threadIdx.x; e < e1; e += EW_THREADS) {
    const int row = e / B.cols, col = e - row * B.cols;
    const float u = bf16_bits_to_float(xi[static_cast<size_t>(row) * B.ld + col]);
    xo[static_cast<size_t>(row) * B.out_ld + col] = static_cast<uint16_t>(float_to_bf16_bits(s * u));
  }
}

// pitch ld -> pitch out_ld copy of bf16 matrices
__global__ void __launch_bounds__(EW_THREADS) unpack_kernel(const __grid_constant__ EwParams p) {
  const EwBank& B = p.b[ew_bank(p)];
  const int local = blockIdx.x - B.block_begin;
  const int mat = local / B.P, chunk = local - mat * B.P;
  const int E = B.rows * B.cols;
  const int e0 = chunk * EW_CHUNK, e1 = min(E, e0 + EW_CHUNK);
  const uint16_t* xi = B.xin + static_cast<size_t>(mat) * B.rows * B.ld;
  uint16_t* xo = B.xout + static_cast<size_t>(mat) * B.rows * B.out_ld;
  for (int e = e0 + threadIdx.x; e < e1; e += EW_THREADS) {
    const int row = e / B.cols, col = e - row * B.cols;
    xo[static_cast<size_t>(row) * B.out_ld + col] = xi[static_cast<size_t>(row) * B.ld + col];
  }
}

// ---------------------------------------------------------------- small-matrix NS (fp32)

constexpr int SMALL_THREADS = 512;

// One block per matrix.  IN_SMEM: both fp32 copies of X and A, B live in
// dynamic shared memory (the gate matrices); otherwise X ping-pongs through the
// fp32 workspace and A, B use the first 2 * SMALL_M^2 floats of shared memory.
template <bool IN_SMEM>
__global__ void __launch_bounds__(SMALL_THREADS) small_ns_kernel(const __grid_constant__ SmallParams p) {
  extern __shared__ float dsm[];
  int bi = 0;
  while (bi + 1 < p.nb && static_cast<int>(blockIdx.x) >= p.b[bi + 1].block_begin) ++bi;
  const SmallBank& B = p.b[bi];
  const int mat = blockIdx.x - B.block_begin;
  const int rows = B.rows, cols = B.cols, E = rows * cols;
  const bool tall = rows > cols;
  const int m = tall ? cols : rows;
  const int n = tall ? rows : cols;
  const size_t moff = static_cast<size_t>(mat) * E;
  float* xf[2];
  float* sA;
  if (IN_SMEM) {
    xf[0] = dsm;
    xf[1] = dsm + E;
    sA = dsm + 2 * E;
  } else {
    xf[0] = B.xf0 + moff;
    xf[1] = B.xf1 + moff;
    sA = dsm;
  }
  float* sB = sA + m * m;
  const uint16_t* x0 = B.x0 + static_cast<size_t>(mat) * rows * B.ld;
  const float s = B.scale[mat];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int e = threadIdx.x; e < E; e += SMALL_THREADS) {
    const int r = e / cols, c = e - r * cols;
    xf[0][e] = s * bf16_bits_to_float(x0[static_cast<size_t>(r) * B.ld + c]);
  }
  __syncthreads();

  // logical X is m x n: X(i, k) = stored(i, k) if wide, stored(k, i) if tall
  for (int it = 0; it < p.steps; ++it) {
    const float* cur = xf[it & 1];
    float* nxt = xf[(it + 1) & 1];
    // A = X X^T (upper triangle, mirrored)
    const int npairs = m * (m + 1) / 2;
    for (int pr = warp; pr < npairs; pr += SMALL_THREADS / 32) {
      int i = 0, rem = pr;
      while (rem >= m - i) {
        rem -= m - i;
        ++i;
      }
      const int j = i + rem;
      float acc = 0.f;
      for (int k = lane; k < n; k += 32) {
        const float xi = tall ? cur[static_cast<size_t>(k) * cols + i] : cur[static_cast<size_t>(i) * cols + k];
        const float xj = tall ? cur[static_cast<size_t>(k) * cols + j] : cur[static_cast<size_t>(j) * cols + k];
        acc = fmaf(xi, xj, acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) {
        sA[i * m + j] = acc;
        sA[j * m + i] = acc;
      }
    }
    __syncthreads();
    // B = b A + c A A
    for (int e = threadIdx.x; e < m * m; e += SMALL_THREADS) {
      const int i = e / m, j = e - i * m;
      float acc = 0.f;
      for (int l = 0; l < m; ++l) acc = fmaf(sA[i * m + l], sA[l * m + j], acc);
      sB[e] = p.cb[it] * sA[e] + p.cc[it] * acc;
    }
    __syncthreads();
    // X <- a X + B X, written in the stored orientation
    for (int e = threadIdx.x; e < E; e += SMALL_THREADS) {
      const int r = e / cols, c = e - r * cols;
      float acc = 0.f;
      if (tall) {  // logical (i = c, k = r): sum_j B[c][j] X(j, r) = sum_j B[c][j] stored(r, j)
        const float* xr = cur + static_cast<size_t>(r) * cols;
        for (int j = 0; j < m; ++j) acc = fmaf(sB[c * m + j], xr[j], acc);
      } else {     // logical (i = r, k = c): sum_j B[r][j] stored(j, c)
        for (int j = 0; j < m; ++j) acc = fmaf(sB[r * m + j], cur[static_cast<size_t>(j) * cols + c], acc);
      }
      nxt[e] = fmaf(p.ca[it], cur[e], acc);
    }
    __syncthreads();
  }
  const float* fin = xf[p.steps & 1];
  uint16_t* out = B.out + static_cast<size_t>(mat) * rows * B.ld;
  for (int e = threadIdx.x; e < E; e += SMALL_THREADS) {
    const int r = e / cols, c = e - r * cols;
    out[static_cast<size_t>(r) * B.ld + c] = static_cast<uint16_t>(float_to_bf16_bits(fin[e]));
  }
}

// ---------------------------------------------------------------- NorMuon row statistics

__global__ void __launch_bounds__(256) row_sumsq_kernel(const __grid_constant__ RowParams p) {
  const int gr = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gr >= p.total_rows) return;
  int bi = 0;
  while (bi + 1 < p.nb && gr >= p.b[bi + 1].row_begin) ++bi;
  const RowBank& B = p.b[bi];
  const int lr = gr - B.row_begin;            // row index over the bank, mat * rows + row
  const int mat = lr / B.rows, row = lr - mat * B.rows;
  const uint16_t* v = B.v + (static_cast<size_t>(mat) * B.rows + row) * B.ld;
  float t = 0.f;
  if ((B.cols & 7) == 0) {
    for (int c = lane * 8; c < B.cols; c += 256) {
      const uint4 w = *reinterpret_cast<const uint4*>(v + c);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = bf16_bits_to_float(ws[i] & 0xFFFFu), b = bf16_bits_to_float(ws[i] >> 16);
        t = fmaf(a, a, t);
        t = fmaf(b, b, t);
      }
    }
  } else {
    for (int c = lane; c < B.cols; c += 32) {
      const float a = bf16_bits_to_float(v[c]);
      t = fmaf(a, a, t);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if (lane == 0) B.q[lr] = t;
}

__global__ void __launch_bounds__(256) row_scale_kernel(const __grid_constant__ RowParams p) {
  __shared__ float red[2][8];
  __shared__ float gshared;
  int bi = 0;
  while (bi + 1 < p.nb && static_cast<int>(blockIdx.x) >= p.b[bi + 1].mat_begin) ++bi;
  const RowBank& B = p.b[bi];
  const int mat = blockIdx.x - B.mat_begin;
  const size_t base = static_cast<size_t>(mat) * B.rows;
  const float inv_cols = 1.0f / static_cast<float>(B.cols);
  const float beta2 = B.dscal ? B.dscal[DSCAL_BETA2] : p.beta2;
  const float b2 = beta2, omb2 = 1.0f - beta2;
  float nv = 0.f, nh = 0.f;
  for (int r = threadIdx.x; r < B.rows; r += 256) {
    float q;
    if (B.rowsq) {
      // the row's sums over its 32-column chunks, written by the Newton-Schulz epilogue, in chunk order
      const float* rq = B.rowsq + static_cast<size_t>(mat) * B.nchunk * B.rows + r;
      q = 0.f;
      for (int c = 0; c < B.nchunk; ++c) q += rq[static_cast<size_t>(c) * B.rows];
      B.q[base + r] = q;
    } else {
      q = B.q[base + r];
    }
    const float s = fmaf(b2, B.state[base + r], omb2 * (q * inv_cols));
    B.state[base + r] = s;
    const float d = fmaxf(s, NORMUON_FLOOR);
    nv += q;
    nh += q / d;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    nv += __shfl_xor_sync(0xffffffffu, nv, o);
    nh += __shfl_xor_sync(0xffffffffu, nh, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = nv;
    red[1][threadIdx.x >> 5] = nh;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f, h = 0.f;
    for (int w = 0; w < 8; ++w) {
      a += red[0][w];
      h += red[1][w];
    }
    gshared = h > 0.f ? sqrtf(a / h) : 0.f;
  }
  __syncthreads();
  const float g = gshared;
  for (int r = threadIdx.x; r < B.rows; r += 256) {
    const float d = fmaxf(B.state[base + r], NORMUON_FLOOR);
    B.rowscale[base + r] = g / sqrtf(d);
  }
}

// ---------------------------------------------------------------- S5 update

template <bool NORMUON>
__global__ void __launch_bounds__(EW_THREADS) k3_kernel(const __grid_constant__ EwParams p) {
  const EwBank& B = p.b[ew_bank(p)];
  const int local = blockIdx.x - B.block_begin;
  const int mat = local / B.P, chunk = local - mat * B.P;
  const int E = B.rows * B.cols;
  const int e0 = chunk * EW_CHUNK, e1 = min(E, e0 + EW_CHUNK);
  const size_t moff = static_cast<size_t>(mat) * E;
  const float decay = B.dscal ? B.dscal[DSCAL_DECAY] : B.decay;
  const float neg_lr = B.dscal ? B.dscal[DSCAL_NEG_LR] : B.neg_lr;
  update_unit<NORMUON>(B.bank + moff, B.mant + moff, B.bank_copy ? B.bank_copy + moff : nullptr,
                       B.xin + static_cast<size_t>(mat) * B.rows * B.ld,
                       NORMUON ? B.rowscale + static_cast<size_t>(mat) * B.rows : nullptr, B.cols, B.ld, e0, e1,
                       threadIdx.x >> 5, threadIdx.x & 31, decay, neg_lr);
}

// ---------------------------------------------------------------- failure-detection self test

__global__ void selftest_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
    // nothing ever arrives on `bar`, so phase 0 never completes
    if (!mbar_wait(&bar, 0, limit_ns)) latch_status(status, DEV_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_k1(const EwParams& p, bool momentum, cudaStream_t s) {
  if (p.total_blocks == 0) return cudaSuccess;
  if (momentum)
    k1_kernel<true><<<p.total_blocks, EW_THREADS, 0, s>>>(p);
  else
    k1_kernel<false><<<p.total_blocks, EW_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_scale(const ScaleParams& p, cudaStream_t s) {
  if (p.total_mats == 0) return cudaSuccess;
  scale_kernel<<<(p.total_mats + 7) / 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_ns0(const EwParams& p, cudaStream_t s) {
  if (p.total_blocks == 0) return cudaSuccess;
  ns0_kernel<<<p.total_blocks, EW_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const EwParams& p, cudaStream_t s) {
  if (p.total_blocks == 0) return cudaSuccess;
  unpack_kernel<<<p.total_blocks, EW_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

long long small_ns_smem_bytes(int rows, int cols) {
  const long long m = rows < cols ? rows : cols;
  return (2ll * rows * cols + 2 * m * m) * static_cast<long long>(sizeof(float));
}

cudaError_t launch_small_ns(const SmallParams& p, bool in_smem, cudaStream_t s) {
  if (p.total_blocks == 0) return cudaSuccess;
  if (!in_smem) {
    small_ns_kernel<false><<<p.total_blocks, SMALL_THREADS, 2 * SMALL_M * SMALL_M * sizeof(float), s>>>(p);
    return cudaGetLastError();
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // set once per device; concurrent first calls from several host threads set it alike
  static std::atomic<bool> attr_done[64];
  if (dev >= 0 && dev < 64 && !attr_done[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(reinterpret_cast<const void*>(small_ns_kernel<true>),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMALL_SMEM_MAX);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  long long bytes = 0;
  for (int i = 0; i < p.nb; ++i) {
    const long long b = small_ns_smem_bytes(p.b[i].rows, p.b[i].cols);
    bytes = b > bytes ? b : bytes;
  }
  if (bytes > SMALL_SMEM_MAX) return cudaErrorInvalidValue;   // such banks take the other path
  small_ns_kernel<true><<<p.total_blocks, SMALL_THREADS, static_cast<size_t>(bytes), s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_row_sumsq(const RowParams& p, cudaStream_t s) {
  if (p.total_rows == 0) return cudaSuccess;
  row_sumsq_kernel<<<(p.total_rows + 7) / 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_row_scale(const RowParams& p, cudaStream_t s) {
  if (p.total_mats == 0) return cudaSuccess;
  row_scale_kernel<<<p.total_mats, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_k3(const EwParams& p, bool normuon, cudaStream_t s) {
  if (p.total_blocks == 0) return cudaSuccess;
  if (normuon)
    k3_kernel<true><<<p.total_blocks, EW_THREADS, 0, s>>>(p);
  else
    k3_kernel<false><<<p.total_blocks, EW_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

// The derived scalars of a step whose hyperparameters sit in device memory: one
// thread per bank forms, in double and rounded once to fp32, exactly what the
// host forms for the by-value calls (1 - mu; 1 - lr*wd as one fused operation;
// -lr times the shape factor), so both kinds of call give identical bits.  An
// invalid value latches DEV_BAD_SCALAR; the step still runs on what it read.
__global__ void scalars_kernel(const __grid_constant__ ScalarParams p) {
  const int i = threadIdx.x;
  if (i >= p.nb) return;
  const ScalarBank& B = p.b[i];
  const float lr = B.src[0], wd = B.src[1], mu = B.src[2], beta2 = B.src[3];
  const bool ok = isfinite(lr) && isfinite(wd) && isfinite(mu) && mu >= 0.f && mu <= 1.f &&
                  (!p.normuon || (isfinite(beta2) && beta2 >= 0.f && beta2 <= 1.f));
  if (!ok) latch_status(p.status, DEV_BAD_SCALAR);
  const double lrd = lr, wdd = wd;
  B.dst[DSCAL_MU] = mu;
  B.dst[DSCAL_OMM] = static_cast<float>(__dsub_rn(1.0, static_cast<double>(mu)));
  B.dst[DSCAL_DECAY] = static_cast<float>(fma(-lrd, wdd, 1.0));
  B.dst[DSCAL_NEG_LR] = static_cast<float>(__dmul_rn(-lrd, B.shape_factor));
  B.dst[DSCAL_BETA2] = beta2;
}

cudaError_t launch_scalars(const ScalarParams& p, cudaStream_t s) {
  if (p.nb <= 0) return cudaSuccess;
  scalars_kernel<<<1, 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace mb
