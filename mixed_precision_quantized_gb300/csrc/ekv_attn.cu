// ekv_attn.cu — single-token GQA decode attention over mixed-format quantized pages.
//
// Computes, for each sequence and query head h with KV head g = h / G,
//   o_h = sum_t softmax_t(sigma q_h . khat_t) vhat_t
// over every cached token ("every decoded token reads the entire KV cache",
// KV-Kaizen, "Background: The KV Cache Bottleneck"), where each page is read
// with its own stored K bit-width ("vLLM's paged attention reads each block
// independently with its stored bit-width", EchoKV, "What happens to old
// blocks when a layer changes tier?") and GQA maps query heads onto KV heads
// (Behavior-Guided KV-Cache Quantization, "Storage savings, with a
// conditional speed trade-off").
//
// Work split: grid (split, kv_head, seq).  A split owns a contiguous range of
// 16-token blocks; each warp of the CTA walks every NW-th block of it.  Per
// block the warp
//   1. loads its slice of the page (codes + scales) with 128/64/32-bit loads,
//   2. unpacks K codes to exact fp16 integers in registers (PRMT/LOP3/HFMA2)
//      and folds the per-channel K scales into Q as an fp16 hi + lo pair,
//   3. S^T[16 tokens x 8 heads] = K . Q^T with mma.sync m16n8k16 (fp32 acc):
//      the block's tokens are M, the GQA group (padded to 8) is N,
//   4. runs the online softmax in the log2 domain, folds each token's V scale
//      into its probability and transposes P with movmatrix,
//   5. O^T[d x 8] += V^T . P^T with mma.sync (channels are M, tokens K).
// Warps merge in shared memory; splits write (max, sum, numerator) partials and
// the last CTA of a (sequence, KV head) — found with an atomic ticket, no
// waiting — merges them by log-sum-exp and writes fp16 O.
#include <math_constants.h>

#include "ekv_internal.h"

namespace ekv {
namespace {

constexpr int NW = 4;  // warps per CTA
constexpr int NT = NW * 32;

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ uint32_t hsub2u(uint32_t a, uint32_t b) {
  return h2u(__hsub2(u2h(a), u2h(b)));
}
__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  return h2u(__hfma2(u2h(a), u2h(b), u2h(c)));
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
  return h2u(__hmul2(u2h(a), u2h(b)));
}

// fp16 bit patterns of constants (exact)
constexpr uint32_t H_1032 = 0x64086408u;   // 1032, 1032
constexpr uint32_t H_1026 = 0x64026402u;   // 1026, 1026
constexpr uint32_t H_1152 = 0x64806480u;   // 1152, 1152
constexpr uint32_t H_MAGIC = 0x64006400u;  // 1024, 1024 exponent pattern

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// ---- K: one row's chunk of KCH = D/4 channels -> KW = KCH/2 half2 words ------
// Word w holds channels (2w, 2w+1) of the chunk as exact fp16 integers q
// (or raw fp16 for 16-bit pages and open-block staging rows).
template <int D>
__device__ __forceinline__ void k_row_words(const uint8_t* row, int kb, int c, uint32_t* kw) {
  constexpr int KCH = D / 4;
  constexpr int KW = KCH / 2;
  if (kb == 4) {
    constexpr int NB = KCH / 2;  // bytes
    uint32_t r[NB / 4];
    if constexpr (NB == 16) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + c * NB));
      r[0] = u.x; r[1] = u.y; r[2] = u.z; r[3] = u.w;
    } else {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(row + c * NB));
      r[0] = u.x; r[1] = u.y;
    }
    const uint32_t mul = 0x2C003C00u;  // (1, 1/16)
    const uint32_t add = 0xD480E408u;  // (-1032, -72)
#pragma unroll
    for (int i = 0; i < NB / 4; ++i)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t t = __byte_perm(r[i], 0, b * 0x1111);
        kw[4 * i + b] = hfma2u(lop3_and_or(t, 0x00F0000Fu, H_MAGIC), mul, add);
      }
  } else if (kb == 2) {
    constexpr int NB = KCH / 4;
    uint32_t r[NB / 4];
    if constexpr (NB == 8) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(row + c * NB));
      r[0] = u.x; r[1] = u.y;
    } else {
      r[0] = __ldg(reinterpret_cast<const uint32_t*>(row + c * NB));
    }
    const uint32_t mul_lo = 0x34003C00u;  // (1, 1/4)
    const uint32_t add_lo = 0xDC08E402u;  // (-1026, -258)
    const uint32_t mul_hi = 0x24002C00u;  // (1/16, 1/64)
    const uint32_t add_hi = 0xCC80D420u;  // (-66, -18)
#pragma unroll
    for (int i = 0; i < NB / 4; ++i)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t t = __byte_perm(r[i], 0, b * 0x1111);
        kw[8 * i + 2 * b] = hfma2u(lop3_and_or(t, 0x000C0003u, H_MAGIC), mul_lo, add_lo);
        kw[8 * i + 2 * b + 1] = hfma2u(lop3_and_or(t, 0x00C00030u, H_MAGIC), mul_hi, add_hi);
      }
  } else if (kb == 8) {
    constexpr int NB = KCH;
#pragma unroll
    for (int i = 0; i < NB / 16; ++i) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + c * NB) + i);
      const uint32_t r[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        kw[8 * i + 2 * x] = hsub2u(__byte_perm(r[x], 0x64646464u, 0x4140), H_1152);
        kw[8 * i + 2 * x + 1] = hsub2u(__byte_perm(r[x], 0x64646464u, 0x4342), H_1152);
      }
    }
  } else {  // raw fp16
#pragma unroll
    for (int i = 0; i < KW / 4; ++i) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + c * KCH * 2) + i);
      kw[4 * i] = u.x; kw[4 * i + 1] = u.y; kw[4 * i + 2] = u.z; kw[4 * i + 3] = u.w;
    }
  }
}

// ---- V: token pair (t, t+1), chunk of VCH = D/8 channels -> VCH words -------
// Word i = (v[t][ch i], v[t+1][ch i]) as exact fp16 integers (raw for 16 bits).
template <int D, int VB>
__device__ __forceinline__ void v_pair_words(const uint8_t* r0, const uint8_t* r1, uint32_t* vw) {
  constexpr int VCH = D / 8;
  constexpr int NB = VCH * VB / 8;  // bytes per row chunk
  constexpr int NWD = NB >= 4 ? NB / 4 : 1;
  uint32_t a[NWD], b[NWD];
  if constexpr (NB == 2) {
    a[0] = __ldg(reinterpret_cast<const uint16_t*>(r0));
    b[0] = __ldg(reinterpret_cast<const uint16_t*>(r1));
  } else if constexpr (NB == 4) {
    a[0] = __ldg(reinterpret_cast<const uint32_t*>(r0));
    b[0] = __ldg(reinterpret_cast<const uint32_t*>(r1));
  } else if constexpr (NB == 8) {
    const uint2 x = __ldg(reinterpret_cast<const uint2*>(r0));
    const uint2 y = __ldg(reinterpret_cast<const uint2*>(r1));
    a[0] = x.x; a[1] = x.y; b[0] = y.x; b[1] = y.y;
  } else {
#pragma unroll
    for (int i = 0; i < NB / 16; ++i) {
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(r0) + i);
      const uint4 y = __ldg(reinterpret_cast<const uint4*>(r1) + i);
      a[4 * i] = x.x; a[4 * i + 1] = x.y; a[4 * i + 2] = x.z; a[4 * i + 3] = x.w;
      b[4 * i] = y.x; b[4 * i + 1] = y.y; b[4 * i + 2] = y.z; b[4 * i + 3] = y.w;
    }
  }
  if constexpr (VB == 4) {
#pragma unroll
    for (int w = 0; w < NWD; ++w) {
      const uint32_t x = __byte_perm(a[w], b[w], 0x5410);
      const uint32_t y = __byte_perm(a[w], b[w], 0x7632);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        vw[8 * w + k] = hsub2u(lop3_and_or(x >> (4 * k), 0x000F000Fu, H_MAGIC), H_1032);
        vw[8 * w + 4 + k] = hsub2u(lop3_and_or(y >> (4 * k), 0x000F000Fu, H_MAGIC), H_1032);
      }
    }
  } else if constexpr (VB == 2) {
    const uint32_t x = __byte_perm(a[0], b[0], 0x5410);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      vw[k] = hsub2u(lop3_and_or(x >> (2 * k), 0x00030003u, H_MAGIC), H_1026);
    if constexpr (VCH == 16) {
      const uint32_t y = __byte_perm(a[0], b[0], 0x7632);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        vw[8 + k] = hsub2u(lop3_and_or(y >> (2 * k), 0x00030003u, H_MAGIC), H_1026);
    }
  } else if constexpr (VB == 8) {
#pragma unroll
    for (int w = 0; w < NWD; ++w)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t x = __byte_perm(a[w], b[w], k | ((4 + k) << 8));
        vw[4 * w + k] = hsub2u(lop3_and_or(x, 0x00FF00FFu, H_MAGIC), H_1152);
      }
  } else {
#pragma unroll
    for (int w = 0; w < NWD; ++w) {
      vw[2 * w] = __byte_perm(a[w], b[w], 0x5410);
      vw[2 * w + 1] = __byte_perm(a[w], b[w], 0x7632);
    }
  }
}

template <int D, int VB>
__global__ void __launch_bounds__(NT)
decode_attn_kernel(DevState st, int layer, const int32_t* __restrict__ slots,
                   const __half* __restrict__ q, __half* __restrict__ o, int splits) {
  constexpr int KCH = D / 4, KW = KCH / 2, NKS = D / 16, VCH = D / 8, NMT = D / 16;
  __shared__ float sm_m[NW][MAX_G], sm_l[NW][MAX_G];
  __shared__ float sm_acc[NW][MAX_G][D];
  __shared__ int s_last;

  const int split = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = st.G;
  const int slot = slots[z];
  const bool slot_ok = slot >= 0 && slot < st.S;
  const int T = slot_ok ? st.len[ls_index(st, layer, slot)] : 0;
  const int nb = (T + BLOCK - 1) / BLOCK;
  const int cb = (nb + splits - 1) / splits;
  const int b0 = min(nb, split * cb), b1 = min(nb, b0 + cb);

  // Q fragment words for head g of the group (zero for padding heads)
  uint32_t qw[KW];
  if (g < G) {
    const uint4* qp = reinterpret_cast<const uint4*>(q + ((size_t)z * st.Hq + h * G + g) * D + c * KCH);
#pragma unroll
    for (int i = 0; i < KW / 4; ++i) {
      const uint4 u = __ldg(qp + i);
      qw[4 * i] = u.x; qw[4 * i + 1] = u.y; qw[4 * i + 2] = u.z; qw[4 * i + 3] = u.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < KW; ++i) qw[i] = 0u;
  }

  float acc[NMT][4];
#pragma unroll
  for (int i = 0; i < NMT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;

  const int32_t* bt = st.bt + lsh_index(st, layer, slot_ok ? slot : 0, h) * st.maxblk;
  const __half* stg = st.staging + lsh_index(st, layer, slot_ok ? slot : 0, h) * (BLOCK * D);
  const float sl = st.scale_log2;

  for (int blk = b0 + warp; blk < b1; blk += NW) {
    const int32_t e = bt[blk];
    if (e == -1) {
      if (lane == 0) set_error(st, EKV_ESTATE);
      continue;
    }
    const int fmt = entry_fmt(e);
    const int kbp = bits_of_code(fmt >> 2);
    const uint8_t* page = st.pool_base[fmt] + (size_t)entry_idx(e) * st.pool_page_bytes[fmt];
    const uint8_t* vpart = page + k_part_bytes(kbp, D);
    const bool open = (blk == nb - 1) && (T % BLOCK != 0);
    const int nv = open ? (T % BLOCK) : BLOCK;

    // ---- S^T = K Q^T ----------------------------------------------------------
    const int kb = open ? 16 : kbp;
    const uint8_t* kbase = open ? reinterpret_cast<const uint8_t*>(stg) : page;
    const int krow = kb == 16 ? 2 * D : D * kb / 8;
    uint32_t kwa[KW], kwb[KW];
    k_row_words<D>(kbase + (size_t)g * krow, kb, c, kwa);
    k_row_words<D>(kbase + (size_t)(g + 8) * krow, kb, c, kwb);
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    if (kb < 16) {
      // Fold the per-channel K scale into Q: q*s = hi + lo with hi = fp16(q*s) and
      // lo = fp16(q*s - hi) from one fused multiply-add (the residual of a rounded
      // fp16 product is itself an fp16 value).  Two MMAs against the exact integer
      // codes keep the logits accurate to fp32 accumulation.
      uint32_t qh[KW], ql[KW];
      const uint4* sp = reinterpret_cast<const uint4*>(page + BLOCK * D * kb / 8 + c * KCH * 2);
#pragma unroll
      for (int i = 0; i < KW / 4; ++i) {
        const uint4 u = __ldg(sp + i);
        const uint32_t sv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          qh[4 * i + x] = hmul2u(qw[4 * i + x], sv[x]);
          ql[4 * i + x] = hfma2u(qw[4 * i + x], sv[x], qh[4 * i + x] ^ 0x80008000u);
        }
      }
#pragma unroll
      for (int kk = 0; kk < NKS; ++kk)
        mma16816(s, kwa[2 * kk], kwb[2 * kk], kwa[2 * kk + 1], kwb[2 * kk + 1], qh[2 * kk],
                 qh[2 * kk + 1]);
#pragma unroll
      for (int kk = 0; kk < NKS; ++kk)
        mma16816(s, kwa[2 * kk], kwb[2 * kk], kwa[2 * kk + 1], kwb[2 * kk + 1], ql[2 * kk],
                 ql[2 * kk + 1]);
    } else {
#pragma unroll
      for (int kk = 0; kk < NKS; ++kk)
        mma16816(s, kwa[2 * kk], kwb[2 * kk], kwa[2 * kk + 1], kwb[2 * kk + 1], qw[2 * kk],
                 qw[2 * kk + 1]);
    }

    // ---- online softmax (log2 domain) -----------------------------------------
    float x0 = s[0] * sl, x1 = s[1] * sl, x2 = s[2] * sl, x3 = s[3] * sl;
    if (g >= nv) x0 = x1 = -CUDART_INF_F;
    if (g + 8 >= nv) x2 = x3 = -CUDART_INF_F;
    float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
    }
    const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
    const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
    l0 = l0 * al0 + (p0 + p2);
    l1 = l1 * al1 + (p1 + p3);
    m0 = mn0;
    m1 = mn1;
#pragma unroll
    for (int i = 0; i < NMT; ++i) {
      acc[i][0] *= al0; acc[i][1] *= al1; acc[i][2] *= al0; acc[i][3] *= al1;
    }

    // ---- P' = P * s_v, transposed into the B fragment --------------------------
    float sv0 = 1.f, sv1 = 1.f;
    if constexpr (VB < 16) {
      const __half* svp = reinterpret_cast<const __half*>(vpart + BLOCK * D * VB / 8);
      sv0 = g < nv ? __half2float(svp[g]) : 0.f;
      sv1 = g + 8 < nv ? __half2float(svp[g + 8]) : 0.f;
    }
    const uint32_t plo = h2u(__floats2half2_rn(p0 * sv0, p1 * sv0));
    const uint32_t phi = h2u(__floats2half2_rn(p2 * sv1, p3 * sv1));
    const uint32_t pb0 = movtrans(plo), pb1 = movtrans(phi);

    // ---- O^T += V^T P^T ---------------------------------------------------------
    constexpr int VROW = VB == 16 ? 2 * D : D * VB / 8;
    constexpr int VOFF = VCH * VB / 8;
    uint32_t va[VCH], vb[VCH];
    const uint8_t* vr = vpart + g * VOFF;
    v_pair_words<D, VB>(vr + (2 * c) * VROW, vr + (2 * c + 1) * VROW, va);
    v_pair_words<D, VB>(vr + (2 * c + 8) * VROW, vr + (2 * c + 9) * VROW, vb);
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt)
      mma16816(acc[mt], va[mt], va[NMT + mt], vb[mt], vb[NMT + mt], pb0, pb1);
  }

  // ---- merge the warps of this CTA ---------------------------------------------
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  if (g == 0) {
    sm_m[warp][2 * c] = m0; sm_m[warp][2 * c + 1] = m1;
    sm_l[warp][2 * c] = l0; sm_l[warp][2 * c + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt) {
    sm_acc[warp][2 * c][g * VCH + mt] = acc[mt][0];
    sm_acc[warp][2 * c + 1][g * VCH + mt] = acc[mt][1];
    sm_acc[warp][2 * c][g * VCH + NMT + mt] = acc[mt][2];
    sm_acc[warp][2 * c + 1][g * VCH + NMT + mt] = acc[mt][3];
  }
  __syncthreads();

  const size_t pbase = ((size_t)z * st.Hkv + h) * splits;
  const size_t pid = pbase + split;
  for (int i = tid; i < G * D; i += NT) {
    const int hd = i / D, ch = i % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w][hd]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = sm_m[w][hd] == -CUDART_INF_F ? 0.f : exp2f(sm_m[w][hd] - M);
      L += f * sm_l[w][hd];
      A += f * sm_acc[w][hd][ch];
    }
    if (splits == 1) {
      o[((size_t)z * st.Hq + h * G + hd) * D + ch] = __float2half_rn(L > 0.f ? A / L : 0.f);
    } else {
      st.attn_acc[(pid * G + hd) * D + ch] = A;
      if (ch == 0) {
        st.attn_ml[(pid * G + hd) * 2] = M;
        st.attn_ml[(pid * G + hd) * 2 + 1] = L;
      }
    }
  }
  if (splits == 1) return;

  // ---- last CTA of this (seq, kv head) merges the splits -------------------------
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int* tk = st.attn_ticket + (size_t)z * st.Hkv + h;
    const int t = atomicAdd(tk, 1);
    s_last = (t == splits - 1);
    if (s_last) *tk = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int i = tid; i < G * D; i += NT) {
    const int hd = i / D, ch = i % D;
    float M = -CUDART_INF_F;
    for (int j = 0; j < splits; ++j) M = fmaxf(M, __ldcg(st.attn_ml + ((pbase + j) * G + hd) * 2));
    float L = 0.f, A = 0.f;
    for (int j = 0; j < splits; ++j) {
      const float mj = __ldcg(st.attn_ml + ((pbase + j) * G + hd) * 2);
      if (mj == -CUDART_INF_F) continue;
      const float f = exp2f(mj - M);
      L += f * __ldcg(st.attn_ml + ((pbase + j) * G + hd) * 2 + 1);
      A += f * __ldcg(st.attn_acc + ((pbase + j) * G + hd) * D + ch);
    }
    o[((size_t)z * st.Hq + h * G + hd) * D + ch] = __float2half_rn(L > 0.f ? A / L : 0.f);
  }
}

template <int D, int VB>
cudaError_t launch_t(const DevState& st, int layer, int n_seqs, const int32_t* slots,
                     const __half* q, __half* o, int splits, cudaStream_t s) {
  dim3 grid(splits, st.Hkv, n_seqs);
  decode_attn_kernel<D, VB><<<grid, NT, 0, s>>>(st, layer, slots, q, o, splits);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attn(const DevState& st, int layer, int n_seqs, const int32_t* slots,
                               const __half* q, __half* o, int splits, int vb, cudaStream_t s) {
  if (st.D == 64) {
    switch (vb) {
      case 2: return launch_t<64, 2>(st, layer, n_seqs, slots, q, o, splits, s);
      case 4: return launch_t<64, 4>(st, layer, n_seqs, slots, q, o, splits, s);
      case 8: return launch_t<64, 8>(st, layer, n_seqs, slots, q, o, splits, s);
      default: return launch_t<64, 16>(st, layer, n_seqs, slots, q, o, splits, s);
    }
  }
  switch (vb) {
    case 2: return launch_t<128, 2>(st, layer, n_seqs, slots, q, o, splits, s);
    case 4: return launch_t<128, 4>(st, layer, n_seqs, slots, q, o, splits, s);
    case 8: return launch_t<128, 8>(st, layer, n_seqs, slots, q, o, splits, s);
    default: return launch_t<128, 16>(st, layer, n_seqs, slots, q, o, splits, s);
  }
}

}  // namespace ekv
