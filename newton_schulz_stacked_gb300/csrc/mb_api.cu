// C ABI of libmuonbank.so: argument checks, workspace layout, TMA tensor
// maps and the launch sequence of one Muon step (S1..S6 of muonbank.h).
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "mb_device.cuh"
#include "mb_internal.h"
#include "muonbank.h"

namespace mb {
namespace {

// Quintic coefficients ("Muon Custom Sizing" write-up, section 2.3).
constexpr float NS_A = 3.4445f, NS_B = -4.7750f, NS_C = 2.0315f;
constexpr size_t WS_ALIGN = 1024;

__device__ int g_status;  // latched device-side status, one per device

thread_local std::string g_last_cuda_error;
thread_local uint64_t g_launch_count = 0;

// Optional stage-boundary events (mb_timing_begin / mb_timing_end).
struct Timing {
  bool on = false;
  int cap = 0, used = 0;
  std::vector<cudaEvent_t> ev;
  std::vector<int> label;
  ~Timing() {   // a thread that ends between mb_timing_begin and mb_timing_end
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
};
thread_local Timing g_timing;

void mark(int label, cudaStream_t st) {
  Timing& t = g_timing;
  if (!t.on || t.used >= t.cap) return;
  if (cudaEventRecord(t.ev[t.used], st) == cudaSuccess) t.label[t.used++] = label;
}

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = cudaGetErrorString(e);
  return MB_ERR_CUDA;
}

#define MB_TRY_CUDA(expr)                      \
  do {                                         \
    cudaError_t e_ = (expr);                   \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)

// A kernel launch: check it, count it and mark its end.
#define MB_LAUNCH(expr, launched, label, stream) \
  do {                                           \
    MB_TRY_CUDA(expr);                           \
    if (launched) {                              \
      ++g_launch_count;                          \
      mark((label), (stream));                   \
    }                                            \
  } while (0)

#define MB_TRY(expr)         \
  do {                       \
    int r_ = (expr);         \
    if (r_ != MB_OK) return r_; \
  } while (0)

// ---------------------------------------------------------------- per-device state

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool ready = false;
  int* status = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[64];

// A second stream per device and host thread on which the fp32 small-matrix
// Newton-Schulz runs beside the tensor-core launch (forked from and joined back
// to the caller's stream with events, so stream order is unchanged).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  // released when the host thread ends; work already queued on the stream still completes
  ~SideStream() {
    if (join) cudaEventDestroy(join);
    if (fork) cudaEventDestroy(fork);
    if (stream) cudaStreamDestroy(stream);
  }
};
thread_local SideStream t_side[64];

int side_stream(SideStream** out) {
  int dev = 0;
  MB_TRY_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MB_ERR_UNSUPPORTED;
  SideStream& s = t_side[dev];
  if (!s.stream) {
    MB_TRY_CUDA(cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking));
    MB_TRY_CUDA(cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming));
    MB_TRY_CUDA(cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming));
  }
  *out = &s;
  return MB_OK;
}
EncodeTiledFn g_encode = nullptr;

int device_state(DeviceState** out) {
  int dev = 0;
  MB_TRY_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    MB_TRY_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    MB_TRY_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
    if (major != 10 || minor != 3) return MB_ERR_UNSUPPORTED;
    void* p = nullptr;
    MB_TRY_CUDA(cudaGetSymbolAddress(&p, g_status));
    d.status = static_cast<int*>(p);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      MB_TRY_CUDA(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
      if (q != cudaDriverEntryPointSuccess || !fn) return MB_ERR_UNSUPPORTED;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  *out = &d;
  return MB_OK;
}

// ---------------------------------------------------------------- checks

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(const mb_shape& s) {
  if (s.batch <= 0 || s.rows <= 0 || s.cols <= 0) return MB_ERR_SHAPE;
  const long long e = static_cast<long long>(s.rows) * s.cols;
  if (e > (1ll << 30)) return MB_ERR_SHAPE;                       // per-matrix element count
  if (static_cast<long long>(s.batch) * e > (1ll << 40)) return MB_ERR_SHAPE;
  const long long blocks = static_cast<long long>(s.batch) * ((e + EW_CHUNK - 1) / EW_CHUNK);
  if (blocks > (1ll << 30)) return MB_ERR_SHAPE;
  if (static_cast<long long>(s.batch) * s.rows > (1ll << 30)) return MB_ERR_SHAPE;
  return MB_OK;
}

int check_ptr(const void* p) {
  if (!p) return MB_ERR_NULL;
  if (!aligned16(p)) return MB_ERR_ALIGN;
  return MB_OK;
}

int check_scalars(float lr, float wd, float mu, float beta2) {
  if (!std::isfinite(lr) || !std::isfinite(wd) || !std::isfinite(mu) || !std::isfinite(beta2)) return MB_ERR_ARG;
  if (mu < 0.f || mu > 1.f || beta2 < 0.f || beta2 > 1.f) return MB_ERR_ARG;
  return MB_OK;
}

// ---------------------------------------------------------------- workspace layout

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
  int batch, rows, cols, m, n, tall, small, ld, ldm, P;
  size_t x[3], a, b, xf[2], partials, scale, q, rowscale;  // x[0] = u, x[1], x[2] = iterates
  size_t rowsq;              // NorMuon, large banks: row sums of v^2 per 32-column chunk [batch][nchunk][rows]
  int nchunk;
  size_t sync, sync_bytes;   // large banks: NS completion counters, then the task counter
  size_t dscal;              // derived scalars of a step with device-memory hyperparameters
  size_t end;
};

Layout make_layout(const mb_shape& s, int normuon, size_t base) {
  Layout L{};
  L.batch = s.batch;
  L.rows = s.rows;
  L.cols = s.cols;
  L.tall = s.rows > s.cols;
  L.m = L.tall ? s.cols : s.rows;
  L.n = L.tall ? s.rows : s.cols;
  L.small = L.m <= SMALL_M;
  // large banks: a multiple of 64 columns, so that an MN-major operand box of 64-column chunks stays in its row
  L.ld = static_cast<int>(align_up(static_cast<size_t>(s.cols), L.small ? 8 : 64));
  L.ldm = static_cast<int>(align_up(static_cast<size_t>(L.m), 8));
  const size_t E = static_cast<size_t>(s.rows) * s.cols;
  L.P = static_cast<int>((E + EW_CHUNK - 1) / EW_CHUNK);
  size_t off = base;
  auto take = [&](size_t bytes) {
    off = align_up(off, WS_ALIGN);
    const size_t r = off;
    off += bytes;
    return r;
  };
  const size_t B = static_cast<size_t>(s.batch);
  for (int i = 0; i < 3; ++i) L.x[i] = take(B * s.rows * L.ld * 2);
  if (!L.small) {
    L.a = take(B * L.m * L.ldm * 2);
    L.b = take(B * L.m * L.ldm * 2);
    L.sync_bytes = B * MAX_NS_STEPS * 3 * sizeof(unsigned) + 16;
    L.sync = take(L.sync_bytes);
  } else {
    L.xf[0] = take(B * E * 4);
    L.xf[1] = take(B * E * 4);
  }
  L.dscal = take(DSCAL_COUNT * sizeof(float));
  L.partials = take(B * L.P * 4);
  L.scale = take(B * 4);
  L.nchunk = (s.cols + 31) / 32;
  if (normuon) {
    L.q = take(B * s.rows * 4);
    L.rowscale = take(B * s.rows * 4);
    if (!L.small) L.rowsq = take(B * static_cast<size_t>(L.nchunk) * s.rows * 4);
  }
  L.end = align_up(off, WS_ALIGN);
  return L;
}

// u stays in x[0]; the iterates X_1, X_2, ... alternate between x[1] and x[2].
int iterate_buffer(int k) { return k == 0 ? 0 : 1 + ((k - 1) & 1); }
int final_buffer(int ns_steps) { return ns_steps == 0 ? 1 : iterate_buffer(ns_steps); }

// ---------------------------------------------------------------- one bank of a step

struct Bank {
  uint16_t* bank;
  uint16_t* bank_copy;  // optional second destination of the updated bank
  int fin = FIN_NONE;   // what the last Newton-Schulz step's epilogue does for this bank (FinMode)
  float decay = 0.f, neg_lr = 0.f;   // S5 scalars (FIN_UPDATE)
  const float* dscal = nullptr;      // or the derived scalars in device memory
  const uint16_t* grad;
  float* mom;
  uint16_t* mant;
  float* row_state;
  Layout L;
  uint8_t* ws;
  template <typename T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(ws + off);
  }
};

int encode_map(CUtensorMap* map, const void* base, int inner, int rows, int batch, int ld, int box_inner,
               int box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2,
                                 static_cast<cuuint64_t>(ld) * static_cast<cuuint64_t>(rows) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = "cuTensorMapEncodeTiled failed (" + std::to_string(static_cast<int>(r)) + ")";
    return MB_ERR_CUDA;
  }
  return MB_OK;
}

// MN-major view of a bf16 buffer of `batch` matrices of `rows` x `ld` (ld a multiple of 64):
// {64 columns, rows, ld / 64 chunks, matrix}; one box is 64 rows of `chunks` 64-column chunks,
// landing chunk after chunk (8 KB each) in the 128-byte swizzle.
int encode_mn_map(CUtensorMap* map, const void* base, int rows, int batch, int ld, int chunks) {
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(ld / 64),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(ld) * 2, 128,
                                 static_cast<cuuint64_t>(ld) * static_cast<cuuint64_t>(rows) * 2};
  const cuuint32_t box[4] = {64, 64, static_cast<cuuint32_t>(chunks), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = "cuTensorMapEncodeTiled (4-D) failed (" + std::to_string(static_cast<int>(r)) + ")";
    return MB_ERR_CUDA;
  }
  return MB_OK;
}

// Element-wise parameter block over a list of banks.
template <typename Fill>
EwParams ew_params(const Bank* banks, int nb, Fill fill) {
  EwParams p{};
  p.nb = nb;
  int blocks = 0;
  for (int i = 0; i < nb; ++i) {
    EwBank& e = p.b[i];
    const Layout& L = banks[i].L;
    e.batch = L.batch;
    e.rows = L.rows;
    e.cols = L.cols;
    e.ld = L.ld;
    e.out_ld = L.ld;
    e.P = L.P;
    e.block_begin = blocks;
    fill(banks[i], e);
    blocks += L.batch * L.P;
  }
  p.total_blocks = blocks;
  return p;
}

// ---------------------------------------------------------------- stages

// S1 (+ S2 partials): u into x[0]; `src_dense` replaces the gradient with a
// ready u when `momentum` is false (the stand-alone NS entry point).
int stage_k1(const Bank* b, int nb, bool momentum, float mu, cudaStream_t st, DeviceState* ds,
             bool dev_scalars = false) {
  EwParams p = ew_params(b, nb, [&](const Bank& k, EwBank& e) {
    e.src = k.grad;
    e.mom = k.mom;
    e.xout = k.at<uint16_t>(k.L.x[0]);
    e.partials = k.at<float>(k.L.partials);
    e.dscal = dev_scalars ? k.at<float>(k.L.dscal) : nullptr;
  });
  p.mu = mu;
  p.omm = static_cast<float>(1.0 - static_cast<double>(mu));
  p.status = ds->status;
  MB_LAUNCH(launch_k1(p, momentum, st), p.total_blocks > 0, MB_MARK_MOMENTUM, st);
  ScaleParams sp{};
  sp.nb = nb;
  int mats = 0;
  for (int i = 0; i < nb; ++i) {
    sp.b[i].partials = b[i].at<float>(b[i].L.partials);
    sp.b[i].scale = b[i].at<float>(b[i].L.scale);
    sp.b[i].batch = b[i].L.batch;
    sp.b[i].P = b[i].L.P;
    sp.b[i].mat_begin = mats;
    mats += b[i].L.batch;
  }
  sp.total_mats = mats;
  MB_LAUNCH(launch_scale(sp, st), sp.total_mats > 0, MB_MARK_SCALE, st);
  return MB_OK;
}

// Each step's (a, b, c): coeffs[3 i .. 3 i + 2] for step i, or the quintic of the pages
// ("Muon Custom Sizing", section 2.3) for every step when coeffs is null.
void set_coeffs(float* ca, float* cb, float* cc, int steps, const float* coeffs) {
  for (int i = 0; i < MAX_NS_STEPS; ++i) {
    const bool own = coeffs && i < steps;
    ca[i] = own ? coeffs[3 * i] : NS_A;
    cb[i] = own ? coeffs[3 * i + 1] : NS_B;
    cc[i] = own ? coeffs[3 * i + 2] : NS_C;
  }
}

int stage_ns_launches(const Bank* b, int nb, int steps, cudaStream_t st, DeviceState* ds, const float* coeffs,
                      SideStream* side, int n_small);

// S3-S4 for every bank: the result lands in x[final_buffer(steps)].
int stage_ns(const Bank* b, int nb, int steps, cudaStream_t st, DeviceState* ds,
             const float* coeffs = nullptr) {
  if (steps == 0) {
    EwParams p = ew_params(b, nb, [&](const Bank& k, EwBank& e) {
      e.xin = k.at<uint16_t>(k.L.x[0]);
      e.xout = k.at<uint16_t>(k.L.x[1]);
      e.scale = k.at<float>(k.L.scale);
    });
    p.status = ds->status;
    MB_LAUNCH(launch_ns0(p, st), p.total_blocks > 0, MB_MARK_NS0, st);
    return MB_OK;
  }
  int n_small = 0, n_large = 0;
  for (int i = 0; i < nb; ++i) (b[i].L.small ? n_small : n_large) += 1;
  // with tensor-core work to overlap, the fp32 small matrices run on the side stream
  SideStream* side = nullptr;
  if (n_small > 0 && n_large > 0) {
    MB_TRY(side_stream(&side));
    MB_TRY_CUDA(cudaEventRecord(side->fork, st));
    MB_TRY_CUDA(cudaStreamWaitEvent(side->stream, side->fork, 0));
  }
  const int r = stage_ns_launches(b, nb, steps, st, ds, coeffs, side, n_small);
  // the caller's stream waits for the side stream on every path, so that nothing launched
  // there outlives the call in stream order, even when a later launch failed
  if (side) {
    const cudaError_t e1 = cudaEventRecord(side->join, side->stream);
    const cudaError_t e2 = e1 == cudaSuccess ? cudaStreamWaitEvent(st, side->join, 0) : e1;
    if (r == MB_OK && e2 != cudaSuccess) return cuda_fail(e2);
  }
  return r;
}

// The launches of stage_ns after the fork of the side stream (null when unused).
int stage_ns_launches(const Bank* b, int nb, int steps, cudaStream_t st, DeviceState* ds, const float* coeffs,
                      SideStream* side, int n_small) {
  // small matrices: fp32 SIMT path; one launch for those whose iteration fits in
  // shared memory, one for the rest
  for (int pass = 0; pass < 2 && n_small > 0; ++pass) {
    const bool in_smem = pass == 0;
    SmallParams sp{};
    sp.steps = steps;
    set_coeffs(sp.ca, sp.cb, sp.cc, steps, coeffs);
    int blocks = 0, n = 0;
    for (int i = 0; i < nb; ++i) {
      const Layout& L = b[i].L;
      if (!L.small) continue;
      if ((small_ns_smem_bytes(L.rows, L.cols) <= SMALL_SMEM_MAX) != in_smem) continue;
      SmallBank& s = sp.b[n++];
      s.x0 = b[i].at<uint16_t>(L.x[0]);
      s.xf0 = b[i].at<float>(L.xf[0]);
      s.xf1 = b[i].at<float>(L.xf[1]);
      s.out = b[i].at<uint16_t>(L.x[final_buffer(steps)]);
      s.scale = b[i].at<float>(L.scale);
      s.batch = L.batch;
      s.rows = L.rows;
      s.cols = L.cols;
      s.ld = L.ld;
      s.block_begin = blocks;
      blocks += L.batch;
    }
    sp.nb = n;
    sp.total_blocks = blocks;
    if (side) {
      MB_TRY_CUDA(launch_small_ns(sp, in_smem, side->stream));
      if (sp.total_blocks > 0) ++g_launch_count;       // no mark: marks time the caller's stream
    } else {
      MB_LAUNCH(launch_small_ns(sp, in_smem, st), sp.total_blocks > 0, MB_MARK_SMALL_NS, st);
    }
  }
  // large matrices: every step of every bank in one fused tcgen05 launch (up to MAX_NS_BANKS banks each)
  int large[MAX_BANKS], nl = 0;
  for (int i = 0; i < nb; ++i)
    if (!b[i].L.small) large[nl++] = i;
  // longest tiles first: the persistent GEMM CTAs take tiles round-robin in this order
  for (int i = 1; i < nl; ++i)
    for (int j = i; j > 0 && b[large[j]].L.n > b[large[j - 1]].L.n; --j) {
      const int t = large[j];
      large[j] = large[j - 1];
      large[j - 1] = t;
    }
  for (int g0 = 0; g0 < nl; g0 += MAX_NS_BANKS) {
    const int gn = (nl - g0 < MAX_NS_BANKS) ? nl - g0 : MAX_NS_BANKS;
    NsParams np{};
    np.nbank = gn;
    np.steps = steps;
    set_coeffs(np.ca, np.cb, np.cc, steps, coeffs);
    np.status = ds->status;
    for (int j = 0; j < gn; ++j) {
      const Bank& k = b[large[g0 + j]];
      const Layout& L = k.L;
      NsBank& nb_ = np.bank[j];
      for (int t = 0; t < 3; ++t) {
        MB_TRY(encode_map(&nb_.xk[t], k.ws + L.x[t], L.cols, L.rows, L.batch, L.ld, 64, 128));
        MB_TRY(encode_mn_map(&nb_.xmn2[t], k.ws + L.x[t], L.rows, L.batch, L.ld, 2));
        MB_TRY(encode_map(&nb_.st_x[t], k.ws + L.x[t], L.cols, L.rows, L.batch, L.ld, 32, 32,
                          CU_TENSOR_MAP_SWIZZLE_64B));
      }
      MB_TRY(encode_map(&nb_.ak, k.ws + L.a, L.m, L.m, L.batch, L.ldm, 64, 128));
      MB_TRY(encode_map(&nb_.bk, k.ws + L.b, L.m, L.m, L.batch, L.ldm, 64, 128));
      MB_TRY(encode_map(&nb_.st_a, k.ws + L.a, L.m, L.m, L.batch, L.ldm, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B));
      MB_TRY(encode_map(&nb_.st_b, k.ws + L.b, L.m, L.m, L.batch, L.ldm, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B));
      nb_.scale = k.at<float>(L.scale);
      nb_.done = k.at<unsigned>(L.sync);
      nb_.fin = k.fin;
      nb_.store_v = 1;
      nb_.w = k.bank;
      nb_.mant = k.mant;
      nb_.w_copy = k.bank_copy;
      nb_.decay = k.decay;
      nb_.neg_lr = k.neg_lr;
      nb_.dscal = k.dscal;
      nb_.rowsq = k.fin == FIN_ROWSQ ? k.at<float>(L.rowsq) : nullptr;
      nb_.nchunk = L.nchunk;
      nb_.batch = L.batch;
      nb_.rows = L.rows;
      nb_.cols = L.cols;
      nb_.m = L.m;
      nb_.n = L.n;
      nb_.tall = L.tall;
      // pair tasks: 256 x 256 tiles of A and B on or above the diagonal, 256 x 256 tiles of X'
      nb_.T = (L.m + 127) / 128;
      const int P2 = (nb_.T + 1) / 2;
      nb_.sym_pairs = P2 * (P2 + 1) / 2;
      const int M = L.tall ? L.n : L.m, N = L.tall ? L.m : L.n;
      nb_.tn = (N + 255) / 256;
      nb_.apply_pairs = ((M + 255) / 256) * nb_.tn;
      MB_TRY_CUDA(cudaMemsetAsync(k.ws + L.sync, 0, L.sync_bytes, st));
    }
    // task numbering inside one step: phase, then bank, then matrix and tile
    int per_iter = 0;
    np.nseg = 0;
    for (int ph = EPI_GRAM; ph <= EPI_APPLY; ++ph) {
      for (int j = 0; j < gn; ++j) {
        np.seg_begin[np.nseg] = per_iter;
        np.seg_bank[np.nseg] = static_cast<unsigned char>(j);
        np.seg_ph[np.nseg] = static_cast<unsigned char>(ph);
        ++np.nseg;
        per_iter += np.bank[j].batch * (ph == EPI_APPLY ? np.bank[j].apply_pairs : np.bank[j].sym_pairs);
      }
    }
    np.seg_begin[np.nseg] = per_iter;
    np.tasks_per_iter = per_iter;
    np.total_tasks = per_iter * steps;
    const Bank& first = b[large[g0]];
    np.next_task = reinterpret_cast<unsigned*>(first.ws + first.L.sync + first.L.sync_bytes - 16);
    MB_LAUNCH(launch_ns_fused(np, st), np.total_tasks > 0, MB_MARK_NS_GEMM, st);
  }
  return MB_OK;
}

// S6 statistics: per-row factor into rowscale, state in place; v with pitch `vld`.  Banks whose
// last Newton-Schulz epilogue wrote their row sums (FIN_ROWSQ) skip the pass over v.
int stage_normuon(const Bank* b, int nb, float beta2, const uint16_t* const* v, const int* vld, cudaStream_t st,
                  bool dev_scalars = false) {
  RowParams rp{}, sp{};
  rp.nb = nb;
  rp.beta2 = sp.beta2 = beta2;
  int rows = 0, mats = 0, srows = 0;
  for (int i = 0; i < nb; ++i) {
    RowBank& r = rp.b[i];
    const Layout& L = b[i].L;
    r.v = v[i];
    r.q = b[i].at<float>(L.q);
    r.rowsq = b[i].fin == FIN_ROWSQ ? b[i].at<float>(L.rowsq) : nullptr;
    r.nchunk = L.nchunk;
    r.state = b[i].row_state;
    r.rowscale = b[i].at<float>(L.rowscale);
    r.batch = L.batch;
    r.rows = L.rows;
    r.cols = L.cols;
    r.ld = vld[i];
    r.row_begin = rows;
    r.mat_begin = mats;
    r.dscal = dev_scalars ? b[i].at<float>(L.dscal) : nullptr;
    rows += L.batch * L.rows;
    mats += L.batch;
    if (!r.rowsq) {
      sp.b[sp.nb] = r;
      sp.b[sp.nb].row_begin = srows;
      ++sp.nb;
      srows += L.batch * L.rows;
    }
  }
  rp.total_rows = rows;
  rp.total_mats = mats;
  sp.total_rows = srows;
  MB_LAUNCH(launch_row_sumsq(sp, st), sp.total_rows > 0, MB_MARK_ROWSTATS, st);
  MB_LAUNCH(launch_row_scale(rp, st), rp.total_mats > 0, MB_MARK_ROWSTATS, st);
  return MB_OK;
}

// S5: update from v (pitch vld); NorMuon uses the per-row factors.  Banks whose last
// Newton-Schulz epilogue already updated them (FIN_UPDATE) are left out.
// sqrt(max(1, rows / cols)): the shape factor of the learning rate ("Muon Custom Sizing", section 4).
double shape_factor(const Layout& L) { return std::sqrt(std::fmax(1.0, static_cast<double>(L.rows) / L.cols)); }

// 1 - lr*wd (rounded once) and -lr*sqrt(max(1, rows/cols)), formed in double and rounded to fp32.
void update_scalars(float lr, float wd, const Layout& L, float* decay, float* neg_lr) {
  const double lrd = lr, wdd = wd;
  *decay = static_cast<float>(std::fma(-lrd, wdd, 1.0));
  *neg_lr = static_cast<float>(-lrd * shape_factor(L));
}

int stage_k3(const Bank* b_all, int nb_all, bool normuon, float lr, float wd, const uint16_t* const* v_all,
             const int* vld_all, cudaStream_t st, bool dev_scalars = false) {
  Bank b[MAX_BANKS];
  const uint16_t* v[MAX_BANKS];
  int vld[MAX_BANKS], nb = 0;
  for (int i = 0; i < nb_all; ++i) {
    if (b_all[i].fin == FIN_UPDATE) continue;
    b[nb] = b_all[i];
    v[nb] = v_all[i];
    vld[nb] = vld_all[i];
    ++nb;
  }
  if (nb == 0) return MB_OK;
  EwParams p = ew_params(b, nb, [&](const Bank& k, EwBank& e) {
    e.bank = k.bank;
    e.bank_copy = k.bank_copy;
    e.mant = k.mant;
    e.rowscale = normuon ? k.at<float>(k.L.rowscale) : nullptr;
    update_scalars(lr, wd, k.L, &e.decay, &e.neg_lr);
    e.dscal = dev_scalars ? k.at<float>(k.L.dscal) : nullptr;
  });
  for (int i = 0; i < nb; ++i) {
    p.b[i].xin = v[i];
    p.b[i].ld = vld[i];
  }
  MB_LAUNCH(launch_k3(p, normuon, st), p.total_blocks > 0, MB_MARK_UPDATE, st);
  return MB_OK;
}

// What the last Newton-Schulz step's epilogue of a bank does in a whole step, as the call's
// MB_STEP_* flags ask: with NorMuon, sum v^2 per row (MB_STEP_FUSE_ROWSTATS); without, apply
// the update itself (MB_STEP_FUSE_UPDATE, rows of whole 16-byte pieces).  Neither for the fp32
// small-matrix path, nor with fewer than 3 steps (the first two steps' APPLY epilogues carry the
// first iterate's residual).
int fin_mode(const Layout& L, int ns_steps, int normuon, unsigned flags) {
  if (L.small || ns_steps < 3) return FIN_NONE;
  if (normuon) return (flags & MB_STEP_FUSE_ROWSTATS) ? FIN_ROWSQ : FIN_NONE;
  return ((flags & MB_STEP_FUSE_UPDATE) && L.cols % 8 == 0) ? FIN_UPDATE : FIN_NONE;
}

// ---------------------------------------------------------------- whole step

int validate_bank(const mb_bank_desc& d, int normuon) {
  MB_TRY(check_shape(d.shape));
  MB_TRY(check_ptr(d.bank));
  MB_TRY(check_ptr(d.grad));
  MB_TRY(check_ptr(d.momentum));
  MB_TRY(check_ptr(d.mantissa));
  if (normuon) MB_TRY(check_ptr(d.row_state));
  if (d.bank_copy && !aligned16(d.bank_copy)) return MB_ERR_ALIGN;
  return MB_OK;
}

// The banks of one call share each launch, whose grid and per-launch counts of
// matrices and rows are 32-bit: together they stay within what one bank may hold.
int check_totals(const Layout* L, int nb) {
  long long blocks = 0, mats = 0, rows = 0;
  for (int i = 0; i < nb; ++i) {
    blocks += static_cast<long long>(L[i].batch) * L[i].P;
    mats += L[i].batch;
    rows += static_cast<long long>(L[i].batch) * L[i].rows;
  }
  return (blocks > (1ll << 30) || mats > (1ll << 30) || rows > (1ll << 30)) ? MB_ERR_SHAPE : MB_OK;
}

int workspace_for(const mb_bank_desc* d, int nb, int normuon, Layout* L, size_t* total) {
  size_t off = 0;
  for (int i = 0; i < nb; ++i) {
    L[i] = make_layout(d[i].shape, normuon, off);
    off = L[i].end;
  }
  MB_TRY(check_totals(L, nb));
  *total = off;
  return MB_OK;
}

int check_workspace(void* ws, size_t have, size_t need) {
  if (!ws) return MB_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MB_ERR_ALIGN;
  if (have < need) return MB_ERR_WORKSPACE;
  return MB_OK;
}

// One step over nb banks.  With `scalars_dev` the hyperparameters are read from
// device memory when the step runs ({lr, wd, mu, beta2} per bank) and lr..beta2
// are ignored.
int run_step(const mb_bank_desc* d, int nb, float lr, float wd, float mu, int normuon, float beta2, int ns_steps,
             void* workspace, size_t ws_bytes, void* stream, const float* scalars_dev = nullptr, unsigned flags = 0) {
  if (!d) return MB_ERR_NULL;
  if (flags & ~static_cast<unsigned>(MB_STEP_FUSE_UPDATE | MB_STEP_FUSE_ROWSTATS)) return MB_ERR_ARG;
  if (nb <= 0 || nb > MAX_BANKS) return nb <= 0 ? MB_ERR_ARG : MB_ERR_TOO_MANY;
  if (ns_steps < 0 || ns_steps > MAX_NS_STEPS) return MB_ERR_NS_STEPS;
  const bool dev = scalars_dev != nullptr;
  if (!dev) MB_TRY(check_scalars(lr, wd, mu, normuon ? beta2 : 0.f));
  for (int i = 0; i < nb; ++i) MB_TRY(validate_bank(d[i], normuon));
  Layout L[MAX_BANKS];
  size_t need = 0;
  MB_TRY(workspace_for(d, nb, normuon, L, &need));
  MB_TRY(check_workspace(workspace, ws_bytes, need));
  DeviceState* ds = nullptr;
  MB_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Bank b[MAX_BANKS];
  const uint16_t* v[MAX_BANKS];
  int vld[MAX_BANKS];
  for (int i = 0; i < nb; ++i) {
    b[i].bank = static_cast<uint16_t*>(d[i].bank);
    b[i].bank_copy = static_cast<uint16_t*>(d[i].bank_copy);
    b[i].grad = static_cast<const uint16_t*>(d[i].grad);
    b[i].mom = d[i].momentum;
    b[i].mant = d[i].mantissa;
    b[i].row_state = d[i].row_state;
    b[i].L = L[i];
    b[i].ws = static_cast<uint8_t*>(workspace);
    b[i].fin = fin_mode(L[i], ns_steps, normuon, flags);
    update_scalars(lr, wd, L[i], &b[i].decay, &b[i].neg_lr);
    b[i].dscal = dev ? b[i].at<float>(L[i].dscal) : nullptr;
    v[i] = b[i].at<uint16_t>(L[i].x[final_buffer(ns_steps)]);
    vld[i] = L[i].ld;
  }
  mark(MB_MARK_BEGIN, st);
  if (dev) {
    // the derived scalars of every bank, read from the caller's buffer as this step runs
    // (timed with the momentum stage)
    ScalarParams sp{};
    sp.nb = nb;
    sp.normuon = normuon;
    sp.status = ds->status;
    for (int i = 0; i < nb; ++i) {
      sp.b[i].src = scalars_dev + 4 * i;
      sp.b[i].dst = b[i].at<float>(L[i].dscal);
      sp.b[i].shape_factor = shape_factor(L[i]);
    }
    MB_TRY_CUDA(launch_scalars(sp, st));
    ++g_launch_count;
  }
  MB_TRY(stage_k1(b, nb, true, mu, st, ds, dev));
  MB_TRY(stage_ns(b, nb, ns_steps, st, ds));
  if (normuon) MB_TRY(stage_normuon(b, nb, beta2, v, vld, st, dev));
  MB_TRY(stage_k3(b, nb, normuon != 0, lr, wd, v, vld, st, dev));
  return MB_OK;
}

// S2-S4 as a stage of its own: u (dense, bf16) in, v (dense, bf16) out.
int ns_stage(const void* u_bf16, void* v_bf16, mb_shape shape, int ns_steps, const float* coeffs, void* workspace,
             size_t workspace_bytes, void* cuda_stream) {
  MB_TRY(check_shape(shape));
  MB_TRY(check_ptr(u_bf16));
  MB_TRY(check_ptr(v_bf16));
  if (ns_steps < 0 || ns_steps > MAX_NS_STEPS) return MB_ERR_NS_STEPS;
  const Layout L = make_layout(shape, 0, 0);
  MB_TRY(check_workspace(workspace, workspace_bytes, L.end));
  DeviceState* ds = nullptr;
  MB_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  Bank k{};
  k.grad = static_cast<const uint16_t*>(u_bf16);
  k.L = L;
  k.ws = static_cast<uint8_t*>(workspace);
  mark(MB_MARK_BEGIN, st);
  MB_TRY(stage_k1(&k, 1, false, 0.f, st, ds));
  MB_TRY(stage_ns(&k, 1, ns_steps, st, ds, coeffs));
  EwParams p = ew_params(&k, 1, [&](const Bank& bk, EwBank& e) {
    e.xin = bk.at<uint16_t>(bk.L.x[final_buffer(ns_steps)]);
    e.xout = static_cast<uint16_t*>(v_bf16);
    e.out_ld = bk.L.cols;
  });
  MB_LAUNCH(launch_unpack(p, st), p.total_blocks > 0, MB_MARK_NS0, st);
  return MB_OK;
}

}  // namespace
}  // namespace mb

using namespace mb;

extern "C" {

int mb_version(void) { return (1 << 16) | 0; }

const char* mb_status_string(int status) {
  switch (status) {
    case MB_OK: return "ok";
    case MB_ERR_NULL: return "a required pointer is NULL";
    case MB_ERR_SHAPE: return "invalid bank shape";
    case MB_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case MB_ERR_NS_STEPS: return "ns_steps outside 0..16";
    case MB_ERR_WORKSPACE: return "workspace missing or too small";
    case MB_ERR_CUDA: return "CUDA error";
    case MB_ERR_TIMEOUT: return "device-side wait timed out";
    case MB_ERR_ARG: return "invalid scalar argument";
    case MB_ERR_UNSUPPORTED: return "device is not sm_103";
    case MB_ERR_TOO_MANY: return "too many banks in one call";
    case MB_ERR_SCRATCH_LIMIT: return "shape needs more than the fixed no-alloc scratch (MB_NOALLOC_SCRATCH_BYTES)";
    case MB_ERR_DEVICE: return "device-side consistency check failed";
    default: return "unknown status";
  }
}

const char* mb_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

int mb_workspace_bytes(mb_shape shape, int normuon, size_t* out_bytes) {
  if (!out_bytes) return MB_ERR_NULL;
  MB_TRY(check_shape(shape));
  *out_bytes = make_layout(shape, normuon, 0).end;
  return MB_OK;
}

int mb_multi_workspace_bytes(const mb_bank_desc* banks, int n_banks, int normuon, size_t* out_bytes) {
  if (!banks || !out_bytes) return MB_ERR_NULL;
  if (n_banks <= 0) return MB_ERR_ARG;
  if (n_banks > MAX_BANKS) return MB_ERR_TOO_MANY;
  for (int i = 0; i < n_banks; ++i) MB_TRY(check_shape(banks[i].shape));
  Layout L[MAX_BANKS];
  return workspace_for(banks, n_banks, normuon, L, out_bytes);
}

int muon_bank_step(void* bank_bf16, const void* grad_bf16, float* momentum_f32, uint16_t* mantissa,
                   mb_shape shape, float lr, float wd, float mu, int ns_steps, void* workspace,
                   size_t workspace_bytes, void* cuda_stream) {
  mb_bank_desc d{bank_bf16, grad_bf16, momentum_f32, mantissa, nullptr, shape, nullptr};
  return run_step(&d, 1, lr, wd, mu, 0, 0.f, ns_steps, workspace, workspace_bytes, cuda_stream);
}

int normuon_bank_step(void* bank_bf16, const void* grad_bf16, float* momentum_f32, uint16_t* mantissa,
                      float* row_state_f32, mb_shape shape, float lr, float wd, float mu, float beta2,
                      int ns_steps, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  mb_bank_desc d{bank_bf16, grad_bf16, momentum_f32, mantissa, row_state_f32, shape, nullptr};
  return run_step(&d, 1, lr, wd, mu, 1, beta2, ns_steps, workspace, workspace_bytes, cuda_stream);
}

int muon_multi_step(const mb_bank_desc* banks, int n_banks, float lr, float wd, float mu, int normuon,
                    float beta2, int ns_steps, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  return run_step(banks, n_banks, lr, wd, mu, normuon ? 1 : 0, beta2, ns_steps, workspace, workspace_bytes,
                  cuda_stream);
}

int muon_multi_step_ex(const mb_bank_desc* banks, int n_banks, float lr, float wd, float mu, int normuon,
                       float beta2, int ns_steps, unsigned flags, void* workspace, size_t workspace_bytes,
                       void* cuda_stream) {
  return run_step(banks, n_banks, lr, wd, mu, normuon ? 1 : 0, beta2, ns_steps, workspace, workspace_bytes,
                  cuda_stream, nullptr, flags);
}

int muon_multi_step_dev(const mb_bank_desc* banks, int n_banks, const float* scalars_dev, int normuon,
                        int ns_steps, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!scalars_dev) return MB_ERR_NULL;
  if (!aligned16(scalars_dev)) return MB_ERR_ALIGN;
  return run_step(banks, n_banks, 0.f, 0.f, 0.f, normuon ? 1 : 0, 0.f, ns_steps, workspace, workspace_bytes,
                  cuda_stream, scalars_dev);
}

int mb_momentum(const void* grad_bf16, float* momentum_f32, void* u_bf16, mb_shape shape, float mu,
                void* cuda_stream) {
  MB_TRY(check_shape(shape));
  MB_TRY(check_ptr(grad_bf16));
  MB_TRY(check_ptr(momentum_f32));
  MB_TRY(check_ptr(u_bf16));
  MB_TRY(check_scalars(0.f, 0.f, mu, 0.f));
  DeviceState* ds = nullptr;
  MB_TRY(device_state(&ds));
  Bank k{};
  k.grad = static_cast<const uint16_t*>(grad_bf16);
  k.mom = momentum_f32;
  k.L = make_layout(shape, 0, 0);
  EwParams p = ew_params(&k, 1, [&](const Bank& bk, EwBank& e) {
    e.src = bk.grad;
    e.mom = bk.mom;
    e.xout = static_cast<uint16_t*>(u_bf16);
    e.out_ld = bk.L.cols;
    e.partials = nullptr;
  });
  p.mu = mu;
  p.omm = static_cast<float>(1.0 - static_cast<double>(mu));
  p.status = ds->status;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  mark(MB_MARK_BEGIN, st);
  MB_LAUNCH(launch_k1(p, true, st), p.total_blocks > 0, MB_MARK_MOMENTUM, st);
  return MB_OK;
}

int mb_newton_schulz(const void* u_bf16, void* v_bf16, mb_shape shape, int ns_steps, void* workspace,
                     size_t workspace_bytes, void* cuda_stream) {
  return ns_stage(u_bf16, v_bf16, shape, ns_steps, nullptr, workspace, workspace_bytes, cuda_stream);
}

int mb_newton_schulz_coeffs(const void* u_bf16, void* v_bf16, mb_shape shape, int ns_steps, const float* coeffs,
                            void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!coeffs) return MB_ERR_NULL;
  if (ns_steps < 0 || ns_steps > MAX_NS_STEPS) return MB_ERR_NS_STEPS;
  for (int i = 0; i < 3 * ns_steps; ++i)
    if (!std::isfinite(coeffs[i])) return MB_ERR_ARG;
  return ns_stage(u_bf16, v_bf16, shape, ns_steps, coeffs, workspace, workspace_bytes, cuda_stream);
}

int mb_update(void* bank_bf16, uint16_t* mantissa, const void* v_bf16, mb_shape shape, float lr, float wd,
              void* cuda_stream) {
  MB_TRY(check_shape(shape));
  MB_TRY(check_ptr(bank_bf16));
  MB_TRY(check_ptr(mantissa));
  MB_TRY(check_ptr(v_bf16));
  MB_TRY(check_scalars(lr, wd, 0.f, 0.f));
  DeviceState* ds = nullptr;
  MB_TRY(device_state(&ds));
  Bank k{};
  k.bank = static_cast<uint16_t*>(bank_bf16);
  k.mant = mantissa;
  k.L = make_layout(shape, 0, 0);
  const uint16_t* v = static_cast<const uint16_t*>(v_bf16);
  const int vld = shape.cols;
  mark(MB_MARK_BEGIN, static_cast<cudaStream_t>(cuda_stream));
  return stage_k3(&k, 1, false, lr, wd, &v, &vld, static_cast<cudaStream_t>(cuda_stream));
}

int mb_normuon_update(void* bank_bf16, uint16_t* mantissa, const void* v_bf16, float* row_state_f32,
                      mb_shape shape, float lr, float wd, float beta2, void* workspace, size_t workspace_bytes,
                      void* cuda_stream) {
  MB_TRY(check_shape(shape));
  MB_TRY(check_ptr(bank_bf16));
  MB_TRY(check_ptr(mantissa));
  MB_TRY(check_ptr(v_bf16));
  MB_TRY(check_ptr(row_state_f32));
  MB_TRY(check_scalars(lr, wd, 0.f, beta2));
  const Layout L = make_layout(shape, 1, 0);
  MB_TRY(check_workspace(workspace, workspace_bytes, L.end));
  DeviceState* ds = nullptr;
  MB_TRY(device_state(&ds));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  Bank k{};
  k.bank = static_cast<uint16_t*>(bank_bf16);
  k.mant = mantissa;
  k.row_state = row_state_f32;
  k.L = L;
  k.ws = static_cast<uint8_t*>(workspace);
  const uint16_t* v = static_cast<const uint16_t*>(v_bf16);
  const int vld = shape.cols;
  mark(MB_MARK_BEGIN, st);
  MB_TRY(stage_normuon(&k, 1, beta2, &v, &vld, st));
  return stage_k3(&k, 1, true, lr, wd, &v, &vld, st);
}

int mb_workspace_views(mb_shape shape, int normuon, int ns_steps, size_t* u_offset, size_t* v_offset,
                       size_t* row_pitch) {
  if (!u_offset || !v_offset || !row_pitch) return MB_ERR_NULL;
  MB_TRY(check_shape(shape));
  if (ns_steps < 0 || ns_steps > MAX_NS_STEPS) return MB_ERR_NS_STEPS;
  const Layout L = make_layout(shape, normuon, 0);
  *u_offset = L.x[0];
  *v_offset = L.x[final_buffer(ns_steps)];
  *row_pitch = static_cast<size_t>(L.ld);
  return MB_OK;
}

int mb_sync_status(void* cuda_stream) {
  DeviceState* ds = nullptr;
  MB_TRY(device_state(&ds));
  MB_TRY_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)));
  int h = 0;
  MB_TRY_CUDA(cudaMemcpy(&h, ds->status, sizeof(int), cudaMemcpyDeviceToHost));
  const int zero = 0;
  MB_TRY_CUDA(cudaMemcpy(ds->status, &zero, sizeof(int), cudaMemcpyHostToDevice));
  return h == DEV_OK ? MB_OK : h == DEV_TIMEOUT ? MB_ERR_TIMEOUT : h == DEV_BAD_SCALAR ? MB_ERR_ARG : MB_ERR_DEVICE;
}

int mb_selftest_timeout(unsigned limit_us, void* cuda_stream) {
  DeviceState* ds = nullptr;
  MB_TRY(device_state(&ds));
  MB_LAUNCH(launch_selftest_timeout(static_cast<uint64_t>(limit_us) * 1000ull, ds->status,
                                    static_cast<cudaStream_t>(cuda_stream)),
            true, MB_MARK_BEGIN, static_cast<cudaStream_t>(cuda_stream));
  return MB_OK;
}

uint64_t mb_launch_count(void) { return g_launch_count; }

int mb_timing_begin(int max_marks) {
  if (max_marks <= 0) return MB_ERR_ARG;
  Timing& t = g_timing;
  if (t.on) return MB_ERR_ARG;
  t.ev.resize(static_cast<size_t>(max_marks));
  t.label.assign(static_cast<size_t>(max_marks), 0);
  for (int i = 0; i < max_marks; ++i) {
    cudaError_t e = cudaEventCreate(&t.ev[i]);
    if (e != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(t.ev[j]);
      t.ev.clear();
      return cuda_fail(e);
    }
  }
  t.cap = max_marks;
  t.used = 0;
  t.on = true;
  return MB_OK;
}

int mb_timing_end(int cap, int* labels, float* ms, int* n_marks) {
  Timing& t = g_timing;
  if (!t.on) return MB_ERR_ARG;
  t.on = false;
  int status = MB_OK;
  const int n = t.used;
  if (n > 0) {
    const cudaError_t e = cudaEventSynchronize(t.ev[n - 1]);
    if (e != cudaSuccess) status = cuda_fail(e);
  }
  for (int i = 0; i < n && i < cap && status == MB_OK; ++i) {
    if (labels) labels[i] = t.label[i];
    float v = 0.f;
    if (i > 0 && t.label[i] != MB_MARK_BEGIN) {
      const cudaError_t e = cudaEventElapsedTime(&v, t.ev[i - 1], t.ev[i]);
      if (e != cudaSuccess) status = cuda_fail(e);
    }
    if (ms) ms[i] = v;
  }
  if (n_marks) *n_marks = n;
  for (cudaEvent_t ev : t.ev) cudaEventDestroy(ev);
  t.ev.clear();
  t.label.clear();
  t.cap = t.used = 0;
  return status;
}

}  // extern "C"

// ---------------------------------------------------------------- no-alloc Newton-Schulz
//
// For callers that may not allocate device memory: the workspace of
// mb_newton_schulz lives in this fixed device array instead (one per device
// that loads the library, held until the process exits).  Calls share it, so
// calls that overlap on the GPU race; nothing in it needs to start at zero.
static __device__ __align__(256) unsigned char mb_noalloc_scratch[MB_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of the scratch array for the current device, looked up once
// per device with that device current (the host-side symbol is not a device address).
int noalloc_scratch(void** out) {
  int dev = 0;
  MB_TRY_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    MB_TRY_CUDA(cudaGetSymbolAddress(&p, mb_noalloc_scratch));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MB_OK;
}
}  // namespace

extern "C" int mb_newton_schulz_noalloc(const void* u_bf16, void* v_bf16, mb_shape shape, int ns_steps,
                                        void* cuda_stream) {
  MB_TRY(check_shape(shape));
  const Layout L = make_layout(shape, 0, 0);
  if (L.end > static_cast<size_t>(MB_NOALLOC_SCRATCH_BYTES)) return MB_ERR_SCRATCH_LIMIT;
  DeviceState* ds = nullptr;
  MB_TRY(device_state(&ds));
  void* scratch = nullptr;
  MB_TRY(noalloc_scratch(&scratch));
  // the same stage as mb_newton_schulz, with the fixed array as its workspace
  return ns_stage(u_bf16, v_bf16, shape, ns_steps, nullptr, scratch, MB_NOALLOC_SCRATCH_BYTES, cuda_stream);
}
