// The element-wise stages as warp-sized units (the momentum with its sums of u^2,
// the normalisation scale, the update), as the element-wise kernels of
// mb_elementwise.cu run them: one unit per warp, with fixed-order reductions.
//
// A chunk is EW_CHUNK consecutive elements of one matrix (row-major, dense);
// its unit w (of EW_UNITS_PER_CHUNK) is the part warp w of a EW_THREADS-thread block
// takes: with cols a multiple of 8, lane l handles the 8-element pieces
// starting at e0 + (j * EW_THREADS + 32 w + l) * 8 for j = 0 .. EW_SLICES-1;
// otherwise the single elements e0 + 32 w + l + EW_THREADS i.
#pragma once

#include "mb_device.cuh"
#include "mb_internal.h"

namespace mb {

constexpr int EW_UNITS_PER_CHUNK = EW_THREADS / 32;   // warp units of a chunk
constexpr int EW_SLICES = EW_CHUNK / (EW_THREADS * 8);

// S1 on one unit ("Muon Custom Sizing" write-up, section 4: buf <- lerp(buf, g, 1 - mu),
// u <- lerp(g, buf, mu)): momentum in place, u (bf16) into xo with row pitch out_ld.  With
// MOMENTUM false the source is a ready u, copied to xo.  Returns the unit's sum of the
// squares of the bf16 u values (a fixed-order sum: each lane in element order, then a
// butterfly over the warp; every lane holds it).
template <bool MOMENTUM>
__device__ __forceinline__ float momentum_unit(const uint16_t* src, float* mom, uint16_t* xo, int cols, int out_ld,
                                               int e0, int e1, int w, int lane, float mu, float omm) {
  float ss = 0.f;
  auto step = [&](float g, float& b) -> float {
    if (!MOMENTUM) return g;
    const float bn = fmaf(omm, g - b, b);  // lerp(buf, g, 1 - mu)
    b = bn;
    return fmaf(mu, bn - g, g);            // lerp(g, buf_new, mu)
  };
  const int t = 32 * w + lane;
  if ((cols & 7) == 0) {
    // every load of the lane's part of the unit first (they may not move past the u stores,
    // which could alias the gradient), then the arithmetic and stores in element order
    uint4 gl[EW_SLICES];
    float4 ml[EW_SLICES][2];
#pragma unroll
    for (int j = 0; j < EW_SLICES; ++j) {
      const int e = e0 + (j * EW_THREADS + t) * 8;
      if (e < e1) {
        gl[j] = *reinterpret_cast<const uint4*>(src + e);
        if (MOMENTUM) {
          ml[j][0] = *reinterpret_cast<const float4*>(mom + e);
          ml[j][1] = *reinterpret_cast<const float4*>(mom + e + 4);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < EW_SLICES; ++j) {
      const int e = e0 + (j * EW_THREADS + t) * 8;
      if (e >= e1) break;
      const int row = e / cols, col = e - row * cols;
      const uint32_t gw[4] = {gl[j].x, gl[j].y, gl[j].z, gl[j].w};
      float bm[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (MOMENTUM) {
        bm[0] = ml[j][0].x; bm[1] = ml[j][0].y; bm[2] = ml[j][0].z; bm[3] = ml[j][0].w;
        bm[4] = ml[j][1].x; bm[5] = ml[j][1].y; bm[6] = ml[j][1].z; bm[7] = ml[j][1].w;
      }
      uint32_t uw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float g0 = bf16_bits_to_float(gw[i] & 0xFFFFu);
        const float g1 = bf16_bits_to_float(gw[i] >> 16);
        const float u0 = step(g0, bm[2 * i]);
        const float u1 = step(g1, bm[2 * i + 1]);
        const uint32_t b0 = float_to_bf16_bits(u0), b1 = float_to_bf16_bits(u1);
        const float r0 = bf16_bits_to_float(b0), r1 = bf16_bits_to_float(b1);
        ss = fmaf(r0, r0, ss);
        ss = fmaf(r1, r1, ss);
        uw[i] = b0 | (b1 << 16);
      }
      if (MOMENTUM) {
        *reinterpret_cast<float4*>(mom + e) = make_float4(bm[0], bm[1], bm[2], bm[3]);
        *reinterpret_cast<float4*>(mom + e + 4) = make_float4(bm[4], bm[5], bm[6], bm[7]);
      }
      *reinterpret_cast<uint4*>(xo + static_cast<size_t>(row) * out_ld + col) = make_uint4(uw[0], uw[1], uw[2], uw[3]);
    }
  } else {
    for (int e = e0 + t; e < e1; e += EW_THREADS) {
      const int row = e / cols, col = e - row * cols;
      float b = MOMENTUM ? mom[e] : 0.f;
      const float u = step(bf16_bits_to_float(src[e]), b);
      if (MOMENTUM) mom[e] = b;
      const uint32_t ub = float_to_bf16_bits(u);
      const float r = bf16_bits_to_float(ub);
      ss = fmaf(r, r, ss);
      xo[static_cast<size_t>(row) * out_ld + col] = static_cast<uint16_t>(ub);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return ss;
}

// The normalisation scale s = 1/(||u||_F + 1e-7) of one matrix from its chunks' sums (n of
// them): each lane adds every 32nd in order, then a butterfly over the warp; every lane
// returns it.
__device__ __forceinline__ float scale_from_units(const float* part, int n, int lane) {
  float t = 0.f;
  for (int i = lane; i < n; i += 32) t += part[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return 1.0f / (sqrtf(t) + 1e-7f);
}

// S5 on one unit (Track-2 record 7 write-up, section 4.1), given v with row pitch ld; with
// NORMUON, v is first scaled by its row's factor rs[row].  bank_copy (optional) also receives
// the new bank bits.
template <bool NORMUON>
__device__ __forceinline__ void update_unit(uint16_t* wb, uint16_t* mb, uint16_t* wc, const uint16_t* v,
                                            const float* rs, int cols, int ld, int e0, int e1, int w, int lane,
                                            float decay, float neg_lr) {
  const int t = 32 * w + lane;
  if ((cols & 7) == 0) {
    // every load of the lane's part of the unit first (the compiler cannot move loads past the
    // stores, which it must assume may alias them), then the arithmetic and stores in order
    uint4 wl[EW_SLICES], ml[EW_SLICES], vl[EW_SLICES];
#pragma unroll
    for (int j = 0; j < EW_SLICES; ++j) {
      const int e = e0 + (j * EW_THREADS + t) * 8;
      if (e < e1) {
        const int row = e / cols, col = e - row * cols;
        wl[j] = *reinterpret_cast<const uint4*>(wb + e);
        ml[j] = *reinterpret_cast<const uint4*>(mb + e);
        vl[j] = *reinterpret_cast<const uint4*>(v + static_cast<size_t>(row) * ld + col);
      }
    }
#pragma unroll
    for (int j = 0; j < EW_SLICES; ++j) {
      const int e = e0 + (j * EW_THREADS + t) * 8;
      if (e >= e1) break;
      const int row = e / cols;
      const float f = NORMUON ? rs[row] : 1.0f;
      uint32_t wa[4] = {wl[j].x, wl[j].y, wl[j].z, wl[j].w}, ma[4] = {ml[j].x, ml[j].y, ml[j].z, ml[j].w};
      const uint32_t va[4] = {vl[j].x, vl[j].y, vl[j].z, vl[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t w0 = wa[i] & 0xFFFFu, w1 = wa[i] >> 16, m0 = ma[i] & 0xFFFFu, m1 = ma[i] >> 16;
        float v0 = bf16_bits_to_float(va[i] & 0xFFFFu), v1 = bf16_bits_to_float(va[i] >> 16);
        if (NORMUON) {
          v0 = __fmul_rn(v0, f);
          v1 = __fmul_rn(v1, f);
        }
        update_one(w0, m0, v0, decay, neg_lr);
        update_one(w1, m1, v1, decay, neg_lr);
        wa[i] = w0 | (w1 << 16);
        ma[i] = m0 | (m1 << 16);
      }
      const uint4 wn = make_uint4(wa[0], wa[1], wa[2], wa[3]);
      *reinterpret_cast<uint4*>(wb + e) = wn;
      *reinterpret_cast<uint4*>(mb + e) = make_uint4(ma[0], ma[1], ma[2], ma[3]);
      if (wc) *reinterpret_cast<uint4*>(wc + e) = wn;
    }
  } else {
    for (int e = e0 + t; e < e1; e += EW_THREADS) {
      const int row = e / cols, col = e - row * cols;
      uint32_t wi = wb[e], mi = mb[e];
      float vf = bf16_bits_to_float(v[static_cast<size_t>(row) * ld + col]);
      if (NORMUON) vf = __fmul_rn(vf, rs[row]);
      update_one(wi, mi, vf, decay, neg_lr);
      wb[e] = static_cast<uint16_t>(wi);
      mb[e] = static_cast<uint16_t>(mi);
      if (wc) wc[e] = static_cast<uint16_t>(wi);
    }
  }
}

}  // namespace mb
