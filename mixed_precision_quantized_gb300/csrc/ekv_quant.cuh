// ekv_quant.cuh — the cache's symmetric quantizer on the device: V rows (per
// token) and sealed K blocks (per channel over the block's 16 tokens), written
// in the page layout.  Shared by the append kernel and the fused append +
// attention kernel.
//
// Quantizer ("Behavior-Guided KV-Cache Quantization", "K/V Role-Aware Low-Bit
// Quantization": symmetric, K per channel, V per token; KV-Kaizen, "Three
// Non-Eviction Compression Axes", item 3: symmetric uniform):
//   s = fp16_rne(m / qmax) with m = min(absmax of the group, c) (IEEE fp32
//   division), q = clamp(rne(x / s), -qmax, qmax), stored offset binary
//   q + 2^(b-1).  c is the group's frozen clipping threshold, +inf unless a
//   calibration artifact set one ("Behavior-Guided KV-Cache Quantization",
//   "Calibration protocol": selected scales and clipping thresholds are frozen
//   and reused by the cache); with c = +inf the quantizer is the plain one.
// KIVI-style asymmetric variant (ASYM; "EchoKV: watching a language model
// decide its own precision", "Show the math", and its per-token KIVI cache,
// "Upstreaming into vLLM"): lo, hi = group min and max,
//   s = fp16_rne((hi - lo) / (2^b - 1)) (fp32 subtraction, IEEE division),
//   z = lo (fp16, exact), u = clamp(rne((x - z) / s), 0, 2^b - 1) stored as is,
//   the zero points right after the scales.
#pragma once

#include <math_constants.h>

#include "ekv_internal.h"

namespace ekv {
namespace {

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// q = clamp(rne(x / s), -qmax, qmax); IEEE division, RNE conversion.
__device__ __forceinline__ int quant_code(float x, float s, int qm) {
  if (s == 0.f) return 0;
  const int q = __float2int_rn(__fdiv_rn(x, s));
  return min(max(q, -qm), qm);
}

// 8 offset-binary codes of b bits, LSB first, as one little-endian word.
__device__ __forceinline__ void store_codes8(uint8_t* dst, const int* u, int b) {
  if (b == 2) {
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) w |= (uint32_t)u[i] << (2 * i);
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)w;
  } else if (b == 4) {
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) w |= (uint32_t)u[i] << (4 * i);
    *reinterpret_cast<uint32_t*>(dst) = w;
  } else {
    unsigned long long w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) w |= (unsigned long long)u[i] << (8 * i);
    *reinterpret_cast<unsigned long long*>(dst) = w;
  }
}

// Asymmetric code of x: clamp(rne((x - z) / s), 0, L); 0 if s = 0.
__device__ __forceinline__ int quant_code_asym(float x, float z, float s, int L) {
  if (s == 0.f) return 0;
  const int u = __float2int_rn(__fdiv_rn(__fsub_rn(x, z), s));
  return min(max(u, 0), L);
}

// Per-channel fp16 values of thread t's channels 8t .. 8t+7 (K scales or zero
// points) in pair order: within each group of n = 32/kb channels (one 32-bit
// code word) position p holds channel p/2 + (p%2)*n/2; 8-bit pages keep the
// natural order.
template <int D>
__device__ __forceinline__ void store_k_group(__half* dst, const __half* v, int kb, int t) {
  if (kb == 8) {
    *reinterpret_cast<uint4*>(dst + 8 * t) = *reinterpret_cast<const uint4*>(v);
  } else if (kb == 4) {  // group = this thread's 8 channels: 0,4,1,5,2,6,3,7
    __align__(16) __half o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = v[i];
      o[2 * i + 1] = v[i + 4];
    }
    *reinterpret_cast<uint4*>(dst + 8 * t) = *reinterpret_cast<const uint4*>(o);
  } else {  // kb == 2: group of 16 channels = threads 2m, 2m+1
    __half* grp = dst + 16 * (t / 2);
#pragma unroll
    for (int i = 0; i < 8; ++i) grp[2 * i + (t & 1)] = v[i];
  }
}

// One V row (one token of one KV head): absmax over D channels, capped at the
// head's threshold vc, one fp16 scale (ASYM: min and max, a scale and a zero
// point).  Called by a whole warp; lanes < D/8 own 8 channels each.
template <int D, bool ASYM = false>
__device__ void quant_v_row(const __half* src, uint8_t* vpart, int r, int vb, int lane,
                            float vc) {
  constexpr int CH = D / 8;
  uint4 u = make_uint4(0, 0, 0, 0);
  float f[8];
  float m = 0.f, lo = CUDART_INF_F, hi = -CUDART_INF_F;
  if (lane < CH) {
    u = *reinterpret_cast<const uint4*>(src + 8 * lane);
    unpack8(u, f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      m = fmaxf(m, fabsf(f[c]));
      lo = fminf(lo, f[c]);
      hi = fmaxf(hi, f[c]);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    if (ASYM) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, off));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    } else {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    }
  }
  if (lane >= CH) return;
  if (vb == 16) {
    *reinterpret_cast<uint4*>(vpart + (size_t)r * 2 * D + 16 * lane) = u;
    return;
  }
  if (ASYM) {
    const int L = (1 << vb) - 1;
    const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), (float)L));
    const float sf = __half2float(s16);
    int code[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) code[c] = quant_code_asym(f[c], lo, sf, L);
    store_codes8(vpart + (size_t)r * (D * vb / 8) + lane * vb, code, vb);
    if (lane == 0) {
      __half* sc = reinterpret_cast<__half*>(vpart + BLOCK * D * vb / 8);
      sc[r] = s16;
      sc[BLOCK + r] = __float2half_rn(lo);
    }
    return;
  }
  const int qm = (1 << (vb - 1)) - 1;
  const __half s16 = __float2half_rn(__fdiv_rn(fminf(m, vc), (float)qm));
  const float sf = __half2float(s16);
  int code[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) code[c] = quant_code(f[c], sf, qm) + (1 << (vb - 1));
  store_codes8(vpart + (size_t)r * (D * vb / 8) + lane * vb, code, vb);
  if (lane == 0) *reinterpret_cast<__half*>(vpart + BLOCK * D * vb / 8 + 2 * r) = s16;
}

// Seal a full K block: thread t owns channels [8t, 8t+8) over the 16 rows.
// Rows before `told` come from the staging rows, the rest from the input;
// kc holds the head's D per-channel thresholds.
template <int D, bool ASYM = false>
__device__ void seal_k(const __half* stg, const __half* kin, size_t in_row, int j, int told,
                       int kb, uint8_t* kpart, int t, const float* kc) {
  float m[8], lo[8], hi[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    m[c] = 0.f;
    lo[c] = CUDART_INF_F;
    hi[c] = -CUDART_INF_F;
  }
  auto row_ptr = [&](int r) -> const __half* {
    const int p = j * BLOCK + r;
    return p < told ? stg + (size_t)r * D + 8 * t : kin + (size_t)(p - told) * in_row + 8 * t;
  };
  if (kb == 16) {
    for (int r = 0; r < BLOCK; ++r)
      *reinterpret_cast<uint4*>(kpart + (size_t)r * 2 * D + 16 * t) =
          *reinterpret_cast<const uint4*>(row_ptr(r));
    return;
  }
  for (int r = 0; r < BLOCK; ++r) {
    float f[8];
    unpack8(*reinterpret_cast<const uint4*>(row_ptr(r)), f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      m[c] = fmaxf(m[c], fabsf(f[c]));
      lo[c] = fminf(lo[c], f[c]);
      hi[c] = fmaxf(hi[c], f[c]);
    }
  }
  __half* sdst = reinterpret_cast<__half*>(kpart + BLOCK * D * kb / 8);
  if (ASYM) {
    const int L = (1 << kb) - 1;
    float sf[8];
    __align__(16) __half s16[8], z16[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      s16[c] = __float2half_rn(__fdiv_rn(__fsub_rn(hi[c], lo[c]), (float)L));
      sf[c] = __half2float(s16[c]);
      z16[c] = __float2half_rn(lo[c]);
    }
    for (int r = 0; r < BLOCK; ++r) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(row_ptr(r)), f);
      int code[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) code[c] = quant_code_asym(f[c], lo[c], sf[c], L);
      store_codes8(kpart + (size_t)r * (D * kb / 8) + t * kb, code, kb);
    }
    store_k_group<D>(sdst, s16, kb, t);
    store_k_group<D>(sdst + D, z16, kb, t);
    return;
  }
  const int qm = (1 << (kb - 1)) - 1;
  const float4 c0 = *reinterpret_cast<const float4*>(kc + 8 * t);
  const float4 c1 = *reinterpret_cast<const float4*>(kc + 8 * t + 4);
  const float cl[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  float sf[8];
  __align__(16) __half s16[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    s16[c] = __float2half_rn(__fdiv_rn(fminf(m[c], cl[c]), (float)qm));
    sf[c] = __half2float(s16[c]);
  }
  for (int r = 0; r < BLOCK; ++r) {
    float f[8];
    unpack8(*reinterpret_cast<const uint4*>(row_ptr(r)), f);
    int code[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) code[c] = quant_code(f[c], sf[c], qm) + (1 << (kb - 1));
    store_codes8(kpart + (size_t)r * (D * kb / 8) + t * kb, code, kb);
  }
  store_k_group<D>(sdst, s16, kb, t);
}

}  // namespace
}  // namespace ekv
