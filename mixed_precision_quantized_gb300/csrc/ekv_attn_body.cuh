// ekv_attn_body.cuh — single-token GQA decode attention over mixed-format quantized
// pages.  Included by ekv_attn.cu (symmetric pages) and ekv_attn_asym.cu (pages
// of the KIVI-style asymmetric quantizer), each with EKV_ATTN_ASYM set, so the
// two variants compile as separate translation units.
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
// Work split: grid (split, kv_head, seq), one CTA per SM.  A split owns a
// contiguous range of 16-token blocks, streamed through one ring of `ns`
// shared-memory stages per CTA: one TMA bulk copy (cp.async.bulk, completion
// counted on an mbarrier) per page, page j in stage j mod ns, refilled with page
// j + ns by the warp that computed page j, so the CTA's HBM requests stay in
// flight while its warps compute.  Warps take pages two at a time: statically
// (warp w the pairs w, w + NW, ...) when the ring holds two pairs per warp or
// more, else from a counter in shared memory.  Per page the warp
//   1. unpacks K codes to exact fp16 integers in registers (PRMT/LOP3/HFMA2)
//      and folds the per-channel K scales into Q as an fp16 hi + lo pair,
//   2. S^T[16 tokens x 8 heads] = K . Q^T with mma.sync m16n8k16 (fp32 acc):
//      the page's tokens are M, the GQA group (padded to 8) is N,
//   3. runs the online softmax in the log2 domain, folds each token's V scale
//      into its probability and transposes P with movmatrix,
//   4. O^T[d x 8] += V^T . P^T with mma.sync (channels are M, tokens K).
// The still-open last block (raw fp16 K rows in the staging buffer) is read
// straight from global memory, first, by one warp.  Warps merge in shared
// memory; splits write (max, sum, numerator) partials and the last CTA of a
// (sequence, KV head) — found with an atomic ticket, no waiting — merges them by
// log-sum-exp.  With static assignment the fp32 summation order is fixed; with
// the shared counter, which warp takes which page depends on timing, so the
// order (not the set of terms) varies from launch to launch.
//
// Asymmetric pages (KIVI-style: xhat = u * s + z, unsigned codes u, fp16 zero
// point z per group, "EchoKV: watching a language model decide its own
// precision", "Show the math" and "Upstreaming into vLLM") change three
// things: the codes unpack without an offset; each K page adds
// sum_c q_c z_c to all its logits (one more MMA chain, the zero points against
// the plain Q); and each V page adds sum_t p_t z_t to every channel of its
// head (fp32 running sums beside l, added before the warps merge).
#pragma once
#ifndef EKV_ATTN_ASYM
#error "define EKV_ATTN_ASYM (0 or 1) before including ekv_attn_body.cuh"
#endif
#include <math_constants.h>

#include "ekv_internal.h"
#include "ekv_quant.cuh"

#if EKV_ATTN_ASYM
#define EKV_ATTN_FN(name) name##_asym
#else
#define EKV_ATTN_FN(name) name##_sym
#endif

namespace ekv {
namespace {

constexpr bool ASYM = EKV_ATTN_ASYM != 0;

constexpr int RING_MAX = 96;             // stages of a CTA's page ring at most (even)
// Blocks the last split of an overlapped launch takes less (~6 us of a CTA's
// page work: how much later its CTAs get an SM).
constexpr int ATTN_LATE_BLOCKS = 80;
// PACK CTAs per SM (1, or 2 when a launch has more (sequence, KV head) units
// than SMs: then every CTA is resident at once and each SM holds a long and a
// short one instead of running a second wave).  Stage memory: 200 KB per SM
// for the CTA's page ring (quantized V: 16 warps, registers capped at 128;
// FP16 V pages are 3.5x larger and need more registers: 12 warps).  After the
// stages come the split's page-table entries.
template <int VB, int PACK = 1>
struct AttnCfg {
  static constexpr int NW = (VB == 16 ? 12 : 16) / PACK;
  static constexpr int NT = NW * 32;
  static constexpr int STAGE_SMEM = 200 * 1024 / PACK;
  static constexpr int BT_CAP = ATTN_BT_CAP / PACK;
  static constexpr int WARP_BYTES = (STAGE_SMEM / NW) & ~127;
  static constexpr int SMEM = STAGE_SMEM + BT_CAP * 4;
};
constexpr int WAIT_LIMIT = 1 << 22;      // bounded mbarrier polls before giving up

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

// fp16 bit patterns of constants (exact)
constexpr uint32_t H_1032 = 0x64086408u;   // 1032, 1032
constexpr uint32_t H_1026 = 0x64026402u;   // 1026, 1026
constexpr uint32_t H_1152 = 0x64806480u;   // 1152, 1152
constexpr uint32_t H_MAGIC = 0x64006400u;  // 1024, 1024 exponent pattern
constexpr uint32_t H_Q4 = 0x34003400u;     // 1/4
constexpr uint32_t H_Q16 = 0x2C002C00u;    // 1/16
constexpr uint32_t H_Q64 = 0x24002400u;    // 1/64
constexpr uint32_t H_M72 = 0xD480D480u;    // -72  = -(1024 + 16*8)/16
constexpr uint32_t H_M258 = 0xDC08DC08u;   // -258 = -(1024 + 4*2)/4
constexpr uint32_t H_M66 = 0xD420D420u;    // -66  = -(1024 + 16*2)/16
constexpr uint32_t H_M18 = 0xCC80CC80u;    // -18  = -(1024 + 64*2)/64
constexpr uint32_t H_M256 = 0xDC00DC00u;   // -256 = -1024/4
constexpr uint32_t H_M64 = 0xD400D400u;    // -64  = -1024/16
constexpr uint32_t H_M16 = 0xCC00CC00u;    // -16  = -1024/64
// Subtrahends that turn the exponent-trick values into codes: the signed code
// q = u - 2^(b-1) for symmetric pages, the unsigned code u for asymmetric ones.
constexpr uint32_t K4_LO = ASYM ? H_MAGIC : H_1032;
constexpr uint32_t K4_HI = ASYM ? H_M64 : H_M72;
constexpr uint32_t C2_0 = ASYM ? H_MAGIC : H_1026;
constexpr uint32_t C2_1 = ASYM ? H_M256 : H_M258;
constexpr uint32_t C2_2 = ASYM ? H_M64 : H_M66;
constexpr uint32_t C2_3 = ASYM ? H_M16 : H_M18;
constexpr uint32_t K8_SUB = ASYM ? H_MAGIC : H_1152;

// x >> 8 as a multiply-high (runs on the FMA pipe, which has spare issue slots).
__device__ __forceinline__ uint32_t shr8(uint32_t x) { return __umulhi(x, 1u << 24); }

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// 2^x with one MUFU op (flushes results below 2^-126 to zero; inputs are
// max-subtracted logits, so the largest term is exactly 1).
__device__ __forceinline__ float fexp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- mbarrier + TMA bulk copy -----------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Poll the stage barrier for the given phase; false if the bound ran out.  A
// non-blocking test first: a landed page (the common case) costs less that way
// than a first try_wait.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  for (int i = 0; i < WAIT_LIMIT; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// ---- loads from global (last block) or shared memory (pipelined pages) ------------
// The last block is read through L2 (.cg): with the fused append its newest row
// (or the whole sealed page) was written earlier in the same launch.
struct GLd {
  const uint8_t* p;
  __device__ __forceinline__ uint4 v4(int o) const {
    return __ldcg(reinterpret_cast<const uint4*>(p + o));
  }
  __device__ __forceinline__ uint2 v2(int o) const {
    return __ldcg(reinterpret_cast<const uint2*>(p + o));
  }
  __device__ __forceinline__ uint32_t v1(int o) const {
    return __ldcg(reinterpret_cast<const uint32_t*>(p + o));
  }
  __device__ __forceinline__ uint32_t h1(int o) const {
    return __ldcg(reinterpret_cast<const uint16_t*>(p + o));
  }
};
// Shared-memory loads through a pointer into the dynamic shared array: ordinary
// loads the compiler may schedule freely after the stage's mbarrier wait (whose
// asm carries a memory clobber, so no load is hoisted above it).
struct SLd {
  const uint8_t* p;
  __device__ __forceinline__ uint4 v4(int o) const {
    return *reinterpret_cast<const uint4*>(p + o);
  }
  __device__ __forceinline__ uint2 v2(int o) const {
    return *reinterpret_cast<const uint2*>(p + o);
  }
  __device__ __forceinline__ uint32_t v1(int o) const {
    return *reinterpret_cast<const uint32_t*>(p + o);
  }
  __device__ __forceinline__ uint32_t h1(int o) const {
    return *reinterpret_cast<const uint16_t*>(p + o);
  }
};

// ---- K: one row's chunk of KCH = D/4 channels -> KW = KCH/2 half2 words -----------
// Word w holds channels (2w, 2w+1) of the chunk as exact fp16 integers q (or raw
// fp16 for 16-bit pages and open-block staging rows).  `row` is the row's offset.
template <int D, int KB, class LD>
__device__ __forceinline__ void k_row_words(const LD& ld, int row, int c, uint32_t* kw) {
  constexpr int KCH = D / 4;
  constexpr int KW = KCH / 2;
  if constexpr (KB == 4) {
    // Word w holds channels 8w..8w+7; out pairs (k, k+4), k = 0..3, matching the
    // pair order of 4-bit scales.
    constexpr int NB = KCH / 2;  // bytes
    uint32_t r[NB / 4];
    if constexpr (NB == 16) {
      const uint4 u = ld.v4(row + c * NB);
      r[0] = u.x; r[1] = u.y; r[2] = u.z; r[3] = u.w;
    } else {
      const uint2 u = ld.v2(row + c * NB);
      r[0] = u.x; r[1] = u.y;
    }
#pragma unroll
    for (int w = 0; w < NB / 4; ++w) {
      const uint32_t r8 = shr8(r[w]);
      kw[4 * w + 0] = hsub2u(lop3_and_or(r[w], 0x000F000Fu, H_MAGIC), K4_LO);
      kw[4 * w + 1] = hfma2u(lop3_and_or(r[w], 0x00F000F0u, H_MAGIC), H_Q16, K4_HI);
      kw[4 * w + 2] = hsub2u(lop3_and_or(r8, 0x000F000Fu, H_MAGIC), K4_LO);
      kw[4 * w + 3] = hfma2u(lop3_and_or(r8, 0x00F000F0u, H_MAGIC), H_Q16, K4_HI);
    }
  } else if constexpr (KB == 2) {
    // Word w holds channels 16w..16w+15; out pairs (k, k+8), k = 0..7.
    constexpr int NB = KCH / 4;
    uint32_t r[NB / 4];
    if constexpr (NB == 8) {
      const uint2 u = ld.v2(row + c * NB);
      r[0] = u.x; r[1] = u.y;
    } else {
      r[0] = ld.v1(row + c * NB);
    }
#pragma unroll
    for (int w = 0; w < NB / 4; ++w) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t x = h ? shr8(r[w]) : r[w];
        kw[8 * w + 4 * h + 0] = hsub2u(lop3_and_or(x, 0x00030003u, H_MAGIC), C2_0);
        kw[8 * w + 4 * h + 1] = hfma2u(lop3_and_or(x, 0x000C000Cu, H_MAGIC), H_Q4, C2_1);
        kw[8 * w + 4 * h + 2] = hfma2u(lop3_and_or(x, 0x00300030u, H_MAGIC), H_Q16, C2_2);
        kw[8 * w + 4 * h + 3] = hfma2u(lop3_and_or(x, 0x00C000C0u, H_MAGIC), H_Q64, C2_3);
      }
    }
  } else if constexpr (KB == 8) {
    constexpr int NB = KCH;
#pragma unroll
    for (int i = 0; i < NB / 16; ++i) {
      const uint4 u = ld.v4(row + c * NB + 16 * i);
      const uint32_t r[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        kw[8 * i + 2 * x] = hsub2u(__byte_perm(r[x], 0x64646464u, 0x4140), K8_SUB);
        kw[8 * i + 2 * x + 1] = hsub2u(__byte_perm(r[x], 0x64646464u, 0x4342), K8_SUB);
      }
    }
  } else {  // raw fp16
#pragma unroll
    for (int i = 0; i < KW / 4; ++i) {
      const uint4 u = ld.v4(row + c * KCH * 2 + 16 * i);
      kw[4 * i] = u.x; kw[4 * i + 1] = u.y; kw[4 * i + 2] = u.z; kw[4 * i + 3] = u.w;
    }
  }
}

// ---- V: token pair (t, t+1), chunk of VCH = D/8 channels -> VCH words -------------
// Word i = (v[t][ch i], v[t+1][ch i]).  For 4- and 8-bit V the words hold the
// *biased* codes the exponent trick yields, A_i = vmul(i) * q + vbias(i) (exact
// fp16 integers); the bias is removed once per warp at the end (see Acc::ps).
// The bias is ~1024 times a 2-bit code, so fp32 accumulation error would grow by
// that much: 2-bit V words are turned into the exact codes q before the MMA.
// Raw fp16 for 16-bit V.
template <int VB>
__host__ __device__ constexpr bool vbias_trick() { return VB == 4 || VB == 8; }
template <int VB>
__host__ __device__ constexpr float vmul(int i) {
  return VB == 4 ? ((i & 1) ? 16.f : 1.f) : 1.f;
}
template <int VB>
__host__ __device__ constexpr float vbias(int i) {
  // 1024 (the exponent pattern) + vmul(i) * 2^(VB-1) (the code offset; none for
  // the unsigned codes of asymmetric pages)
  return vbias_trick<VB>() ? 1024.f + (ASYM ? 0.f : vmul<VB>(i) * (float)(1 << (VB - 1)))
                           : 0.f;
}

// `flip` (0 or 0x4444) marks lanes that loaded the pair's rows in swapped order
// (row t+1 from offset r0): it swaps the two sources of every byte permute.
template <int D, int VB, class LD>
__device__ __forceinline__ void v_pair_words(const LD& ld, int r0, int r1, uint32_t flip,
                                             uint32_t* vw) {
  constexpr int VCH = D / 8;
  constexpr int NB = VCH * VB / 8;  // bytes per row chunk
  constexpr int NWD = NB >= 4 ? NB / 4 : 1;
  uint32_t a[NWD], b[NWD];
  if constexpr (NB == 2) {
    a[0] = ld.h1(r0);
    b[0] = ld.h1(r1);
  } else if constexpr (NB == 4) {
    a[0] = ld.v1(r0);
    b[0] = ld.v1(r1);
  } else if constexpr (NB == 8) {
    const uint2 x = ld.v2(r0), y = ld.v2(r1);
    a[0] = x.x; a[1] = x.y; b[0] = y.x; b[1] = y.y;
  } else {
#pragma unroll
    for (int i = 0; i < NB / 16; ++i) {
      const uint4 x = ld.v4(r0 + 16 * i), y = ld.v4(r1 + 16 * i);
      a[4 * i] = x.x; a[4 * i + 1] = x.y; a[4 * i + 2] = x.z; a[4 * i + 3] = x.w;
      b[4 * i] = y.x; b[4 * i + 1] = y.y; b[4 * i + 2] = y.z; b[4 * i + 3] = y.w;
    }
  }
  if constexpr (VB == 4) {
#pragma unroll
    for (int w = 0; w < NWD; ++w) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // channels 8w+4h .. 8w+4h+3
        const uint32_t x = __byte_perm(a[w], b[w], (h ? 0x7632u : 0x5410u) ^ flip);
        const uint32_t x8 = shr8(x);
        vw[8 * w + 4 * h + 0] = lop3_and_or(x, 0x000F000Fu, H_MAGIC);
        vw[8 * w + 4 * h + 1] = lop3_and_or(x, 0x00F000F0u, H_MAGIC);
        vw[8 * w + 4 * h + 2] = lop3_and_or(x8, 0x000F000Fu, H_MAGIC);
        vw[8 * w + 4 * h + 3] = lop3_and_or(x8, 0x00F000F0u, H_MAGIC);
      }
    }
  } else if constexpr (VB == 2) {
#pragma unroll
    for (int h = 0; h < VCH / 8; ++h) {  // channels 8h .. 8h+7
      const uint32_t x = __byte_perm(a[0], b[0], (h ? 0x7632u : 0x5410u) ^ flip);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t y = q ? shr8(x) : x;
        vw[8 * h + 4 * q + 0] = hsub2u(lop3_and_or(y, 0x00030003u, H_MAGIC), C2_0);
        vw[8 * h + 4 * q + 1] = hfma2u(lop3_and_or(y, 0x000C000Cu, H_MAGIC), H_Q4, C2_1);
        vw[8 * h + 4 * q + 2] = hfma2u(lop3_and_or(y, 0x00300030u, H_MAGIC), H_Q16, C2_2);
        vw[8 * h + 4 * q + 3] = hfma2u(lop3_and_or(y, 0x00C000C0u, H_MAGIC), H_Q64, C2_3);
      }
    }
  } else if constexpr (VB == 8) {
#pragma unroll
    for (int w = 0; w < NWD; ++w)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t x = __byte_perm(a[w], b[w], (k | ((4 + k) << 8)) ^ flip);
        vw[4 * w + k] = lop3_and_or(x, 0x00FF00FFu, H_MAGIC);
      }
  } else {
#pragma unroll
    for (int w = 0; w < NWD; ++w) {
      vw[2 * w] = __byte_perm(a[w], b[w], 0x5410u ^ flip);
      vw[2 * w + 1] = __byte_perm(a[w], b[w], 0x7632u ^ flip);
    }
  }
}

// Online-softmax state of one warp (per thread: heads 2c, 2c+1 of the group).
// o: O^T fragments (biased for 4- and 8-bit V); ps: running sum of the fp16 P'
// that entered the PV products, per head (C fragment of P'^T summed over its
// 16 rows by an MMA with an all-ones A), used to remove the V code bias.
template <int D>
struct Acc {
  float o[D / 16][4];
  float ps[4];
  float m0, m1, l0, l1;
  float z0, z1;  // asymmetric V: this lane's sum of p_t z_t, heads 2c and 2c+1
};

// K code pairing of a page format: 0 = adjacent channels (8- and 16-bit pages),
// 1 = (k, k+4) within 8 channels (4-bit), 2 = (k, k+8) within 16 channels (2-bit).
template <int KB>
__host__ __device__ constexpr int pair_class() { return KB == 4 ? 1 : KB == 2 ? 2 : 0; }

// Q words of head g over this thread's channel chunk, paired like the K codes of
// pairing class pc (zero for padding heads).
template <int D>
__device__ __forceinline__ void load_q(const __half* qp, bool valid, int pc, uint32_t* qw) {
  constexpr int KW = D / 8;
  uint32_t nat[KW];
  if (valid) {
#pragma unroll
    for (int i = 0; i < KW / 4; ++i) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(qp) + i);
      nat[4 * i] = u.x; nat[4 * i + 1] = u.y; nat[4 * i + 2] = u.z; nat[4 * i + 3] = u.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < KW; ++i) nat[i] = 0u;
  }
  if (pc == 1) {
#pragma unroll
    for (int w = 0; w < KW / 4; ++w)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        qw[4 * w + k] = __byte_perm(nat[4 * w + k / 2], nat[4 * w + 2 + k / 2],
                                    (k & 1) ? 0x7632 : 0x5410);
  } else if (pc == 2) {
#pragma unroll
    for (int w = 0; w < KW / 8; ++w)
#pragma unroll
      for (int k = 0; k < 8; ++k)
        qw[8 * w + k] = __byte_perm(nat[8 * w + k / 2], nat[8 * w + 4 + k / 2],
                                    (k & 1) ? 0x7632 : 0x5410);
  } else {
#pragma unroll
    for (int i = 0; i < KW; ++i) qw[i] = nat[i];
  }
}

// S^T[16 tokens x 8 heads] of one page into s[4] (C fragment: tokens g, g+8 x
// heads 2c, 2c+1).  KB bits (raw fp16 if 16); the K part is read through kl.
template <int D, int KB, class KL>
__device__ __forceinline__ void page_scores(const KL& kl, const uint32_t* qw, float* s, int g,
                                            int c) {
  constexpr int KCH = D / 4, KW = KCH / 2, NKS = D / 16;
  constexpr int krow = KB == 16 ? 2 * D : D * KB / 8;
  uint32_t kwa[KW], kwb[KW];
  k_row_words<D, KB>(kl, g * krow, c, kwa);
  k_row_words<D, KB>(kl, (g + 8) * krow, c, kwb);
  float s1[4] = {0.f, 0.f, 0.f, 0.f};
  s[0] = s[1] = s[2] = s[3] = 0.f;
  if constexpr (KB == 4 || KB == 8 || (ASYM && KB == 2)) {
    // Fold the per-channel K scale into Q: q*s = hi + lo with hi = fp16(q*s) and
    // lo = fp16(q*s - hi) from one fused multiply-add (the residual of a rounded
    // fp16 product is itself an fp16 value).  Two MMA chains against the exact
    // integer codes keep the logits accurate to fp32 accumulation.
    uint32_t qh[KW], ql[KW];
    const int so = BLOCK * D * KB / 8 + c * KCH * 2;
#pragma unroll
    for (int i = 0; i < KW / 4; ++i) {
      const uint4 u = kl.v4(so + 16 * i);
      const uint32_t sv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const __half2 hi = __hmul2(u2h(qw[4 * i + x]), u2h(sv[x]));
        qh[4 * i + x] = h2u(hi);
        ql[4 * i + x] = h2u(__hfma2(u2h(qw[4 * i + x]), u2h(sv[x]), __hneg2(hi)));
      }
    }
#pragma unroll
    for (int kk = 0; kk < NKS; ++kk) {
      mma16816(s, kwa[2 * kk], kwb[2 * kk], kwa[2 * kk + 1], kwb[2 * kk + 1], qh[2 * kk],
               qh[2 * kk + 1]);
      mma16816(s1, kwa[2 * kk], kwb[2 * kk], kwa[2 * kk + 1], kwb[2 * kk + 1], ql[2 * kk],
               ql[2 * kk + 1]);
    }
    if constexpr (ASYM) {
      // sum_c q_c z_c, the same for all 16 tokens: every A row holds the zero
      // points (stored after the scales, in the same order), B is the plain Q.
      const int zo = so + 2 * D;
#pragma unroll
      for (int i = 0; i < KW / 4; ++i) {
        const uint4 u = kl.v4(zo + 16 * i);
        mma16816(s1, u.x, u.x, u.y, u.y, qw[4 * i], qw[4 * i + 1]);
        mma16816(s1, u.z, u.z, u.w, u.w, qw[4 * i + 2], qw[4 * i + 3]);
      }
    }
  } else {
    if constexpr (KB == 2) {
      // 2-bit codes are 0, +-1 or -2, so code times its (pair-ordered) channel
      // scale is exact in fp16: scale the codes and run one MMA chain with plain Q.
      const int so = BLOCK * D * KB / 8 + c * KCH * 2;
#pragma unroll
      for (int i = 0; i < KW / 4; ++i) {
        const uint4 u = kl.v4(so + 16 * i);
        const uint32_t sv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          kwa[4 * i + x] = h2u(__hmul2(u2h(kwa[4 * i + x]), u2h(sv[x])));
          kwb[4 * i + x] = h2u(__hmul2(u2h(kwb[4 * i + x]), u2h(sv[x])));
        }
      }
    }
#pragma unroll
    for (int kk = 0; kk < NKS; kk += 2) {
      mma16816(s, kwa[2 * kk], kwb[2 * kk], kwa[2 * kk + 1], kwb[2 * kk + 1], qw[2 * kk],
               qw[2 * kk + 1]);
      mma16816(s1, kwa[2 * kk + 2], kwb[2 * kk + 2], kwa[2 * kk + 3], kwb[2 * kk + 3],
               qw[2 * kk + 2], qw[2 * kk + 3]);
    }
  }
  s[0] += s1[0]; s[1] += s1[1]; s[2] += s1[2]; s[3] += s1[3];
}

// P' = P * s_v for one page, transposed by movmatrix into the PV B fragment.
template <int D, int VB, class VL>
__device__ __forceinline__ void page_probs(const VL& vl, int nv, float p0, float p1, float p2,
                                           float p3, int g, uint32_t& pb0, uint32_t& pb1,
                                           Acc<D>& A) {
  float sv0 = 1.f, sv1 = 1.f;
  if constexpr (VB < 16) {
    const int so = BLOCK * D * VB / 8;
    const uint32_t w0 = vl.h1(so + 2 * g), w1 = vl.h1(so + 2 * (g + 8));
    sv0 = g < nv ? __half2float(__ushort_as_half((unsigned short)w0)) : 0.f;
    sv1 = g + 8 < nv ? __half2float(__ushort_as_half((unsigned short)w1)) : 0.f;
    if constexpr (ASYM) {  // zero points of tokens g and g+8 (after the 16 scales)
      const uint32_t y0 = vl.h1(so + 32 + 2 * g), y1 = vl.h1(so + 32 + 2 * (g + 8));
      const float z0 = g < nv ? __half2float(__ushort_as_half((unsigned short)y0)) : 0.f;
      const float z1 = g + 8 < nv ? __half2float(__ushort_as_half((unsigned short)y1)) : 0.f;
      A.z0 = fmaf(p0, z0, fmaf(p2, z1, A.z0));
      A.z1 = fmaf(p1, z0, fmaf(p3, z1, A.z1));
    }
  }
  pb0 = movtrans(h2u(__floats2half2_rn(p0 * sv0, p1 * sv0)));
  pb1 = movtrans(h2u(__floats2half2_rn(p2 * sv1, p3 * sv1)));
}

// O^T[d x 8] += V^T P^T for one page.
template <int D, int VB, class VL>
__device__ __forceinline__ void page_pv(const VL& vl, uint32_t pb0, uint32_t pb1, Acc<D>& A,
                                        int g, int c) {
  constexpr int VCH = D / 8, NMT = D / 16;
  constexpr int VROW = VB == 16 ? 2 * D : D * VB / 8;
  constexpr int VOFF = VCH * VB / 8;
  uint32_t va[VCH], vb[VCH];
  // Lanes with odd c read row 2c+1 first: rows 2c of the four c fall on the same
  // banks, so alternating the order halves the bank conflicts of each load.
  const int odd = c & 1;
  const uint32_t flip = odd ? 0x4444u : 0u;
  const int vr = g * VOFF;
  v_pair_words<D, VB>(vl, vr + (2 * c + odd) * VROW, vr + (2 * c + 1 - odd) * VROW, flip, va);
  v_pair_words<D, VB>(vl, vr + (2 * c + 8 + odd) * VROW, vr + (2 * c + 9 - odd) * VROW, flip, vb);
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt)
    mma16816(A.o[mt], va[mt], va[NMT + mt], vb[mt], vb[NMT + mt], pb0, pb1);
  if constexpr (vbias_trick<VB>()) {
    constexpr uint32_t ONES = 0x3C003C00u;  // fp16 (1, 1)
    mma16816(A.ps, ONES, ONES, ONES, ONES, pb0, pb1);
  }
}

// Online-softmax update over up to two pages of the same K width at once (one
// shared max reduction); page b is skipped when nvb == 0.
template <int D, int VB, bool FULL, int KB, class KLA, class VLA, class KLB, class VLB>
__device__ __forceinline__ void attend_pages(const KLA& kla, const VLA& vla, int nva,
                                             const KLB& klb, const VLB& vlb, int nvb,
                                             const uint32_t* qw, Acc<D>& A, float sl, int g,
                                             int c) {
  constexpr int NMT = D / 16;
  float sa[4], sb[4];
  page_scores<D, KB>(kla, qw, sa, g, c);
  if (nvb > 0) page_scores<D, KB>(klb, qw, sb, g, c);
  float xa0 = sa[0] * sl, xa1 = sa[1] * sl, xa2 = sa[2] * sl, xa3 = sa[3] * sl;
  if (!FULL) {  // rows past the valid count carry no token
    if (g >= nva) xa0 = xa1 = -CUDART_INF_F;
    if (g + 8 >= nva) xa2 = xa3 = -CUDART_INF_F;
  }
  float xb0 = -CUDART_INF_F, xb1 = -CUDART_INF_F, xb2 = -CUDART_INF_F, xb3 = -CUDART_INF_F;
  if (nvb > 0) {
    xb0 = sb[0] * sl; xb1 = sb[1] * sl; xb2 = sb[2] * sl; xb3 = sb[3] * sl;
    if (!FULL) {
      if (g >= nvb) xb0 = xb1 = -CUDART_INF_F;
      if (g + 8 >= nvb) xb2 = xb3 = -CUDART_INF_F;
    }
  }
  // Lazy max: the reference A.m moves only when a score passes it by more than
  // SLACK (log2 units), so most pages skip the cross-lane reduction.  Then
  // p = 2^(x - m) <= 2^SLACK, and P' = p * s_v stays below the fp16 maximum for
  // any stored V scale (s_v <= 65504 / qmax).
  constexpr float SLACK = VB == 2 ? 0.f : VB == 4 ? 2.f : VB == 8 ? 6.f : 8.f;
  float bm0 = fmaxf(fmaxf(xa0, xa2), fmaxf(xb0, xb2));
  float bm1 = fmaxf(fmaxf(xa1, xa3), fmaxf(xb1, xb3));
  if (__any_sync(0xffffffffu, bm0 > A.m0 + SLACK || bm1 > A.m1 + SLACK)) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
    }
    const float mn0 = fmaxf(A.m0, bm0), mn1 = fmaxf(A.m1, bm1);
    if (mn0 != A.m0 || mn1 != A.m1) {  // rescale only when a reference moved
      const float al0 = fexp2(A.m0 - mn0), al1 = fexp2(A.m1 - mn1);
      A.l0 *= al0;
      A.l1 *= al1;
      if constexpr (ASYM && VB < 16) {
        A.z0 *= al0;
        A.z1 *= al1;
      }
#pragma unroll
      for (int i = 0; i < NMT; ++i) {
        A.o[i][0] *= al0; A.o[i][1] *= al1; A.o[i][2] *= al0; A.o[i][3] *= al1;
      }
      if constexpr (vbias_trick<VB>()) {
        A.ps[0] *= al0; A.ps[1] *= al1; A.ps[2] *= al0; A.ps[3] *= al1;
      }
      A.m0 = mn0;
      A.m1 = mn1;
    }
  }
  const float mn0 = A.m0, mn1 = A.m1;
  const float pa0 = fexp2(xa0 - mn0), pa1 = fexp2(xa1 - mn1);
  const float pa2 = fexp2(xa2 - mn0), pa3 = fexp2(xa3 - mn1);
  A.l0 += pa0 + pa2;
  A.l1 += pa1 + pa3;
  uint32_t qa0, qa1;
  page_probs<D, VB>(vla, FULL ? BLOCK : nva, pa0, pa1, pa2, pa3, g, qa0, qa1, A);
  if (nvb > 0) {
    const float pb0 = fexp2(xb0 - mn0), pb1 = fexp2(xb1 - mn1);
    const float pb2 = fexp2(xb2 - mn0), pb3 = fexp2(xb3 - mn1);
    A.l0 += pb0 + pb2;
    A.l1 += pb1 + pb3;
    uint32_t qb0, qb1;
    page_probs<D, VB>(vlb, FULL ? BLOCK : nvb, pb0, pb1, pb2, pb3, g, qb0, qb1, A);
    page_pv<D, VB>(vla, qa0, qa1, A, g, c);
    page_pv<D, VB>(vlb, qb0, qb1, A, g, c);
  } else {
    page_pv<D, VB>(vla, qa0, qa1, A, g, c);
  }
}

template <int N>
struct KBits {
  static constexpr int value = N;
};
template <bool B>
struct BoolC {
  static constexpr bool value = B;
};
// Call f(KBits<kb>{}) with the page K width as a compile-time constant.
template <class F>
__device__ __forceinline__ void with_kbits(int kb, F&& f) {
  switch (kb) {
    case 2: f(KBits<2>{}); break;
    case 4: f(KBits<4>{}); break;
    case 8: f(KBits<8>{}); break;
    default: f(KBits<16>{}); break;
  }
}

// A split partial holds the CTA's O^T fragments in "slot" order: element j of
// m-tile mt of lane's fragment goes to slot (mt*4 + j)*32 + lane, so a warp
// stores and loads whole 128-byte rows.  Slot -> (query head of the group, channel):
template <int D>
__device__ __forceinline__ int slot_head(int s) { return 2 * (s & 3) + ((s >> 5) & 1); }
template <int D>
__device__ __forceinline__ int slot_ch(int s) {
  constexpr int VCH = D / 8, NMT = D / 16;
  return ((s & 31) >> 2) * VCH + ((s >> 6) & 1) * NMT + (s >> 7);
}
// Thread t of a CTA of NT threads owns slots t + k*NT (k < PTS); NT is a multiple
// of 64, so they share the slot bits that pick the head: all of head slot_head(t).  MCH partials are loaded per
// merge round, as many as fit the registers without spilling.
template <int D, int NT>
struct MergeShape {
  static_assert(NT % 64 == 0, "slots of a thread must share a head");
  static constexpr int SLOTS = MAX_G * D;
  static constexpr int PTS = (SLOTS + NT - 1) / NT;
  static constexpr int MCH = 80 / (PTS + 2) < 20 ? 80 / (PTS + 2) : 20;
};

// Merge `count` split partials at slots pbase + first + j*stride (j < count) by
// log-sum-exp.  Every thread merges its own slots straight from global memory
// (L2: other CTAs wrote them): the (max, sum) pair of its head and its slot
// values of up to MCH partials are loaded in one round, then folded into a
// running (M, L, acc).  With `orow` set the result is normalized and written to
// O as fp16; otherwise the unnormalized (M, L, values) go to slot `dst`, which
// may be one of the slots read (a barrier separates the reads from the writes).
// Called by every thread of the CTA.
template <int D, int NT>
__device__ __noinline__ void merge_parts(float* __restrict__ part_acc, float* __restrict__ part_ml,
                                         size_t pbase, int first, int stride, int count, int G,
                                         int tid, __half* __restrict__ orow, size_t dst) {
  constexpr int SLOTS = MergeShape<D, NT>::SLOTS, PTS = MergeShape<D, NT>::PTS;
  constexpr int MCH = MergeShape<D, NT>::MCH;
  const int hd = slot_head<D>(tid);
  const bool active = hd < G;  // padding heads of the group are never read
  float M = -CUDART_INF_F, L = 0.f;
  float acc[PTS];
#pragma unroll
  for (int k = 0; k < PTS; ++k) acc[k] = 0.f;
  if (active) {
    const float* accb = part_acc + (pbase + first) * SLOTS + tid;
    const float* mlb = part_ml + ((pbase + first) * MAX_G + hd) * 2;
    const size_t astep = (size_t)stride * SLOTS, mstep = (size_t)stride * MAX_G * 2;
    for (int j0 = 0; j0 < count; j0 += MCH) {
      float2 ml[MCH];
      float a[MCH][PTS];
#pragma unroll
      for (int u = 0; u < MCH; ++u) {
        ml[u] = make_float2(-CUDART_INF_F, 0.f);
#pragma unroll
        for (int k = 0; k < PTS; ++k) a[u][k] = 0.f;
        if (j0 + u < count) {
          ml[u] = __ldcg(reinterpret_cast<const float2*>(mlb + (j0 + u) * mstep));
#pragma unroll
          for (int k = 0; k < PTS; ++k)
            if (tid + k * NT < SLOTS) a[u][k] = __ldcg(accb + (j0 + u) * astep + k * NT);
        }
      }
      float Mn = M;
#pragma unroll
      for (int u = 0; u < MCH; ++u) Mn = fmaxf(Mn, ml[u].x);
      if (Mn == -CUDART_INF_F) continue;  // nothing attended so far
      const float al = M == -CUDART_INF_F ? 0.f : exp2f(M - Mn);
      L *= al;
#pragma unroll
      for (int k = 0; k < PTS; ++k) acc[k] *= al;
#pragma unroll
      for (int u = 0; u < MCH; ++u) {
        const float f = ml[u].x == -CUDART_INF_F ? 0.f : exp2f(ml[u].x - Mn);
        L = fmaf(f, ml[u].y, L);
#pragma unroll
        for (int k = 0; k < PTS; ++k) acc[k] = fmaf(f, a[u][k], acc[k]);
      }
      M = Mn;
    }
  }
  if (orow) {
    if (active) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int k = 0; k < PTS; ++k)
        if (tid + k * NT < SLOTS)
          orow[hd * D + slot_ch<D>(tid + k * NT)] = __float2half_rn(acc[k] * inv);
    }
    return;
  }
  __syncthreads();  // every read of the slots is done before `dst` is overwritten
  if (active) {
#pragma unroll
    for (int k = 0; k < PTS; ++k)
      if (tid + k * NT < SLOTS) part_acc[dst * SLOTS + tid + k * NT] = acc[k];
    if ((tid & ~32) < 4)  // the first thread of each head
      *reinterpret_cast<float2*>(part_ml + (dst * MAX_G + hd) * 2) = make_float2(M, L);
  }
}

// Merge `count` (<= ATTN_GROUP) split partials at slots pbase + j into O, in one
// round of loads: every thread loads its slots of all the partials, while warp w
// < MAX_G loads head w's (max, sum) pairs, reduces them across its lanes and
// leaves the partials' weights 2^(m_j - M) and 1 / L in shared memory
// (s_f[j][head], s_inv[head]); after one barrier each thread folds its slots.
// Called by every thread of the CTA (NT >= MAX_G * 32).
template <int D, int NT>
__device__ __noinline__ void merge_final(const float* __restrict__ part_acc,
                                         const float* __restrict__ part_ml, size_t pbase,
                                         int count, int G, int tid, __half* __restrict__ orow,
                                         float (*s_f)[MAX_G], float* s_inv) {
  constexpr int SLOTS = MergeShape<D, NT>::SLOTS, PTS = MergeShape<D, NT>::PTS;
  static_assert(NT >= MAX_G * 32, "one warp per head of the group");
  const int hd = slot_head<D>(tid);
  const bool active = hd < G;
  float a[ATTN_GROUP][PTS];
#pragma unroll
  for (int j = 0; j < ATTN_GROUP; ++j)
#pragma unroll
    for (int k = 0; k < PTS; ++k)
      a[j][k] = active && j < count && tid + k * NT < SLOTS
                    ? __ldcg(part_acc + (pbase + j) * SLOTS + tid + k * NT)
                    : 0.f;
  const int w = tid >> 5, lane = tid & 31;
  if (w < G) {
    float2 ml = make_float2(-CUDART_INF_F, 0.f);
    if (lane < count)
      ml = __ldcg(reinterpret_cast<const float2*>(part_ml + ((pbase + lane) * MAX_G + w) * 2));
    float M = ml.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float f = ml.x == -CUDART_INF_F ? 0.f : exp2f(ml.x - M);
    float L = f * ml.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane < count) s_f[lane][w] = f;
    if (lane == 0) s_inv[w] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  if (!active) return;
  float acc[PTS];
#pragma unroll
  for (int k = 0; k < PTS; ++k) acc[k] = 0.f;
#pragma unroll
  for (int j = 0; j < ATTN_GROUP; ++j) {
    if (j < count) {
      const float f = s_f[j][hd];
#pragma unroll
      for (int k = 0; k < PTS; ++k) acc[k] = fmaf(f, a[j][k], acc[k]);
    }
  }
  const float inv = s_inv[hd];
#pragma unroll
  for (int k = 0; k < PTS; ++k)
    if (tid + k * NT < SLOTS)
      orow[hd * D + slot_ch<D>(tid + k * NT)] = __float2half_rn(acc[k] * inv);
}

// Arrive on a merge ticket that `expected` CTAs share: publish this CTA's
// writes, count it in, and return (to every thread) whether it came last.  The
// last one resets the ticket for the next launch and sees all the others' writes.
// The barrier orders every thread's writes before thread 0's release; thread 0's
// acquire and the second barrier order the other CTAs' writes before every
// thread's reads (which go through L2: __ldcg).
__device__ __forceinline__ bool last_arrival(int* ticket, int expected, int tid, int* s_flag) {
  __syncthreads();
  if (tid == 0) {
    int t;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(t) : "l"(ticket) : "memory");
    *s_flag = (t == expected - 1);
    if (*s_flag) *ticket = 0;  // the next launch's arrivals come after this launch ends
  }
  __syncthreads();
  return *s_flag != 0;
}

// The fused append of one token, by one warp: the same steps as the append
// kernel for n_new = 1 ("How EchoKV works": the step's K enters the layer's
// FP16 ring and, quantized, the paged cache; "What happens to old blocks when a
// layer changes tier?": a block's page is admitted at the tier current when its
// first token arrives).  Block j receives the token at row r: a page is popped
// when r == 0, the V row is quantized into it, the K row goes to the staging
// rows or, at r == 15, seals the block.  Returns the page entry (-1: none).
template <int D>
__device__ int32_t append_token(const DevState& st, int layer, int slot, int h, int j, int r,
                                int told, const __half* kin, const __half* vin, int lane) {
  constexpr int CH = D / 8;
  int32_t e = -1;
  if (lane == 0) {
    int32_t* btp = st.bt + lsh_index(st, layer, slot, h) * st.maxblk + j;
    if (r == 0) {  // block opens now: admit at the layer's current tier
      const int fmt = code_of_bits(st.tier[layer]) * 4 + code_of_bits(st.vbits[layer]);
      const int old = atomicSub(st.top + fmt, 1);
      if (old <= 0) {
        atomicAdd(st.top + fmt, 1);
        set_error(st, EKV_ENOMEM);
      } else {
        e = (int32_t)(((uint32_t)fmt << 28) | (uint32_t)st.stack[fmt][old - 1]);
        atomicMax(st.kmax + layer, st.tier[layer]);
      }
      *btp = e;
    } else {
      e = *btp;
      if (e == -1) set_error(st, EKV_ESTATE);  // an existing block must have a page
    }
  }
  e = __shfl_sync(0xffffffffu, e, 0);
  const size_t lsh = lsh_index(st, layer, slot, h);
  __half* stg = st.staging + lsh * (BLOCK * D);
  if (e != -1) {
    const int fmt = entry_fmt(e);
    const int kb = bits_of_code(fmt >> 2), vb = bits_of_code(fmt & 3);
    uint8_t* page = st.pool_base[fmt] + (size_t)entry_idx(e) * st.pool_page_bytes[fmt];
    const size_t lh = (size_t)layer * st.Hkv + h;
    quant_v_row<D, ASYM>(vin, page + k_part_bytes(kb, D, ASYM), r, vb, lane, st.vclip[lh]);
    if (r == BLOCK - 1) {
      if (lane < CH) seal_k<D, ASYM>(stg, kin, 0, j, told, kb, page, lane, st.kclip + lh * D);
    } else if (lane < CH) {
      *reinterpret_cast<uint4*>(stg + (size_t)r * D + 8 * lane) =
          *reinterpret_cast<const uint4*>(kin + 8 * lane);
    }
  }
  if (lane < CH)  // ring: the newest 64 K vectors, slot p % 64
    *reinterpret_cast<uint4*>(st.ring + lsh * (RING * D) + (size_t)(told % RING) * D + 8 * lane) =
        *reinterpret_cast<const uint4*>(kin + 8 * lane);
  __syncwarp();  // the block's new bytes are visible to the warp's loads that follow
  return e;
}

template <int D, int VB, bool FUSED, int PACK, bool A_ = ASYM>
__global__ void __launch_bounds__(AttnCfg<VB, PACK>::NT, PACK)
decode_attn_kernel(DevState st, int layer, const int32_t* __restrict__ slots,
                   const __half* __restrict__ q, __half* __restrict__ o, int splits,
                   const __half* __restrict__ knew, const __half* __restrict__ vnew,
                   int late_blocks, int dep_inputs) {
  using Cfg = AttnCfg<VB, PACK>;
  constexpr int NW = Cfg::NW, NT = Cfg::NT;
  constexpr int KCH = D / 4, KW = KCH / 2, NMT = D / 16;
  static_assert(NT >= RING_MAX, "the first ring fill gives each thread one page at most");
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[RING_MAX];
  __shared__ int s_issued[RING_MAX];  // last page copied into each stage (-1: none)
  __shared__ float sm_m[NW][MAX_G], sm_l[NW][MAX_G], sm_f[NW][MAX_G], sm_ml[MAX_G][2];
  __shared__ float sm_mf[ATTN_GROUP][MAX_G], sm_inv[MAX_G];  // final merge weights
  __shared__ int s_next, s_last;
  int32_t* s_bt = reinterpret_cast<int32_t*>(smem + Cfg::STAGE_SMEM);

  // Block order: KV head fastest, then sequence (in the order of `slots`), then
  // split, so the CTAs that start last are the last split of every (sequence,
  // KV head), and a caller that lists its longest sequences first gets them
  // started first (longest-first scheduling of a ragged batch).
  const int n_seqs = gridDim.x / (splits * st.Hkv);
  const int h = blockIdx.x % st.Hkv, z = blockIdx.x / st.Hkv % n_seqs;
  const int split = blockIdx.x / (n_seqs * st.Hkv);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int G = st.G;
  const int slot = slots[z];
  const bool slot_ok = slot >= 0 && slot < st.S;
  const int told = slot_ok ? st.len[ls_index(st, layer, slot)] : 0;
  // Fused append: this launch adds one token to every sequence and attends over
  // it too.  Every CTA reads the old length; the last CTA of the sequence to be
  // done with it publishes the new one (ticket below).
  bool app = false;
  if constexpr (FUSED) {
    if (!slot_ok) {
      if (tid == 0 && split == 0 && h == 0) set_error(st, EKV_EINVAL);
    } else if (told + 1 > st.maxblk * BLOCK) {  // would outgrow the block table
      if (tid == 0 && split == 0 && h == 0) set_error(st, EKV_ESTATE);
    } else {
      app = true;
    }
  }
  const int T = told + (app ? 1 : 0);
  const int nb = (T + BLOCK - 1) / BLOCK;
  // Contiguous block ranges, the last split's `late_blocks` short of an even
  // share: when this launch overlaps the end of the one before (programmatic
  // dependent), the last split's CTAs are the ones that get an SM last, a few
  // microseconds (that launch's final merges) after the others.
  int b0 = 0, b1 = nb;
  if (splits > 1) {
    const int rest = nb - max(0, nb / splits - late_blocks);
    const int cb = (rest + splits - 2) / (splits - 1);
    b0 = split < splits - 1 ? min(rest, split * cb) : rest;
    b1 = split < splits - 1 ? min(rest, b0 + cb) : nb;
  }
  // Sealed blocks of this split go through the pipelines.  The sequence's last
  // block is attended from global memory by the split that holds it when it is
  // open (raw K rows in the staging buffer) or receives this launch's token.
  const bool last_apart = ((T % BLOCK) != 0 || app) && b1 == nb && b1 > b0;
  int np = b1 - b0 - (last_apart ? 1 : 0);  // pipelined pages of this split
  if (np > Cfg::BT_CAP) {  // the host sizes splits so that this never happens
    if (tid == 0) set_error(st, EKV_ESTATE);
    np = 0;
  }

  const int32_t* bt = st.bt + lsh_index(st, layer, slot_ok ? slot : 0, h) * st.maxblk;
  const __half* stg = st.staging + lsh_index(st, layer, slot_ok ? slot : 0, h) * (BLOCK * D);
  // Stage ring of the CTA: ns stages (even, at most RING_MAX) sized for the
  // widest page this layer has admitted so far.  Page j of the split always goes
  // to stage j % ns; its copy is the (j / ns)-th completion of that stage's
  // barrier.  Pages 0 .. ns-1 are copied at the start; the warp that finishes
  // page j copies page j + ns into the stage it just emptied, and records it in
  // s_issued, which the warp that takes page j + ns reads before it waits (so
  // it never waits on a barrier phase other than its page's).
  const int kmax = max(2, st.kmax[layer]);
  const int stage_bytes = (page_bytes(kmax, VB, D, ASYM) + 127) & ~127;
  // Static assignment when the ring holds two pairs per warp or more: warp w
  // takes pairs w, w + NW, ... and ns is a multiple of 2 NW, so page j + ns is
  // the same warp's page as page j and each warp refills only its own stages
  // (no shared counter, no issue check).  Larger pages keep the deeper ring and
  // a shared counter (any warp takes the next pair).
  const int ns_fit = min(RING_MAX, Cfg::STAGE_SMEM / stage_bytes) & ~1;
  const int ns_static = ns_fit / (2 * NW) * (2 * NW);
  // (Launches of two CTAs per SM keep the shared counter: with static assignment
  // their batched, two-wave launches ran up to milliseconds long.)
  const bool stat = PACK == 1 && ns_static >= 4 * NW;
  const int ns = stat ? ns_static : ns_fit;
  // j / ns as a multiply-high (exact for j < 2^32 / ns^2, far above the pages of a split)
  const uint32_t ns_magic = (uint32_t)((0x100000000ull + ns - 1) / ns);
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t bar0 = (uint32_t)__cvta_generic_to_shared(&bars[0]);
  if (tid < ns) {
    mbar_init(bar0 + 8 * tid, 1);
    s_issued[tid] = -1;
  }
  if (tid == 0) asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

  // Copy the split's page-table entries and check whether every pipelined page
  // has one format (the common case: a layer whose tier did not change over the
  // split's range); such a split runs a loop specialized to that format.
  const int32_t e_first = np > 0 ? bt[b0] : -1;
  int mixed = 0;
  for (int i = tid; i < np; i += NT) {
    const int32_t e = bt[b0 + i];
    s_bt[i] = e;
    mixed |= (e == -1) | (((uint32_t)(e ^ e_first) >> 28) != 0);
  }
  if (tid == 0) s_next = 0;

  // Q fragment words for head g of the group, paired like the K codes of the
  // page format in use (re-paired when a page of another pairing class comes);
  // loaded once the first page copies are in flight.
  const __half* qrow = q + ((size_t)z * st.Hq + h * G + (g < G ? g : 0)) * D + c * KCH;
  uint32_t qw[KW];
  int qpc = 0;
  auto pair_q = [&](auto kbc) {
    constexpr int PC = pair_class<decltype(kbc)::value>();
    if (qpc != PC) {
      load_q<D>(qrow, g < G, PC, qw);
      qpc = PC;
    }
  };

  Acc<D> A;
#pragma unroll
  for (int i = 0; i < NMT; ++i) A.o[i][0] = A.o[i][1] = A.o[i][2] = A.o[i][3] = 0.f;
  A.ps[0] = A.ps[1] = A.ps[2] = A.ps[3] = 0.f;
  A.m0 = A.m1 = -CUDART_INF_F;
  A.l0 = A.l1 = 0.f;
  A.z0 = A.z1 = 0.f;
  const float sl = st.scale_log2;

  // page-table copy, counter and barriers ready
  const bool uniform = !__syncthreads_or(mixed) && np > 0 && e_first != -1;

  // A uniform split under static assignment gives each stage pair one barrier
  // (pages k, k + 1 of a warp's pair, k even, in stages si, si + 1 signal
  // barrier si / 2), so its warps wait once per pair.
  const bool pairb = stat && uniform;
  // The pool of a uniform split's pages (its only format).
  const int fmt_u = uniform ? entry_fmt(e_first) : 0;
  const uint32_t bytes_u = (uint32_t)st.pool_page_bytes[fmt_u];
  const uint8_t* base_u = st.pool_base[fmt_u];
  // One thread: page k into stage si (= k % ns).  A page whose table entry is
  // missing (-1) is flagged and not copied, but still completes its barrier
  // phase (an arrival with no bytes), so the stage's phase count stays k / ns.
  // With pair barriers the thread of the even page arrives expecting the bytes
  // of both (the odd page's copy may land first: the transaction count dips
  // below zero, but the phase cannot complete before that arrival).
  auto issue = [&](int k, int si) {
    const int32_t e = s_bt[k];
    uint32_t bytes = 0;
    const uint8_t* src = nullptr;
    if (uniform) {
      bytes = bytes_u;
      src = base_u + (size_t)entry_idx(e) * bytes_u;
    } else if (e != -1) {
      const int fmt = entry_fmt(e);
      bytes = (uint32_t)st.pool_page_bytes[fmt];
      src = st.pool_base[fmt] + (size_t)entry_idx(e) * bytes;
    }
    if (src) {
      const uint32_t bar = bar0 + 8 * (pairb ? si >> 1 : si);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      if (!pairb)
        mbar_expect_tx(bar, bytes);
      else if (!(si & 1))
        mbar_expect_tx(bar, k + 1 < np ? 2 * bytes : bytes);
      bulk_g2s(sbase + si * stage_bytes, src, bytes, bar);
    } else {
      set_error(st, EKV_ESTATE);
      mbar_arrive(bar0 + 8 * si);
    }
    *reinterpret_cast<volatile int*>(&s_issued[si]) = k;
  };
  // The first ns pages, spread over all warps (warp w copies pages w, w + NW, ...;
  // 32 NW >= RING_MAX): a warp's copy instructions go out one issuing lane after
  // another, so a few lanes in each warp finish sooner than 32 lanes in two.
  {
    const int p = warp + NW * lane;
    if (p < ns && p < np) issue(p, p);
  }

  // Dependent-inputs overlap: everything above read only this layer's cache
  // state (length, page table, pages) and the slot list; the launch before may
  // still be writing Q, K and V, so wait for it before the first read of them.
  // Once it is complete, a programmatic dependent of this launch (the next
  // layer's) may start on an SM as soon as this launch's CTA there exits: it
  // reads only its own layer's state before its own wait, and that layer's last
  // writer is at least the launch before this one, now complete.  (A launch
  // triggers only after its own wait, so at most two are ever in flight.  Two
  // CTAs per SM trigger after their loop instead: started early, the next
  // launch's CTAs would fill the SMs in block order and undo the pairing of a
  // long and a short sequence on each SM that a longest-first slot list gives.)
  if (dep_inputs) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (PACK == 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  load_q<D>(qrow, g < G, 0, qw);

  // The last block first (with the fused append, after appending to it), while
  // the first copies are in flight.
  if (last_apart && warp == NW - 1) {
    int32_t e;
    if (app) {
      const size_t in = ((size_t)z * st.Hkv + h) * D;
      e = append_token<D>(st, layer, slot, h, nb - 1, told % BLOCK, told, knew + in, vnew + in,
                          lane);
    } else {
      e = __ldcg(bt + nb - 1);
      if (e == -1 && lane == 0) set_error(st, EKV_ESTATE);
    }
    if (e != -1) {
      const int fmt = entry_fmt(e);
      const uint8_t* page = st.pool_base[fmt] + (size_t)entry_idx(e) * st.pool_page_bytes[fmt];
      const int kb = bits_of_code(fmt >> 2);
      const GLd vl{page + k_part_bytes(kb, D, ASYM)};
      if (T % BLOCK == 0) {  // sealed by this launch's token: a full page
        with_kbits(kb, [&](auto kbc) {
          constexpr int KB = decltype(kbc)::value;
          pair_q(kbc);
          attend_pages<D, VB, true, KB>(GLd{page}, vl, BLOCK, GLd{page}, vl, 0, qw, A, sl, g, c);
        });
      } else {
        const GLd kl{reinterpret_cast<const uint8_t*>(stg)};
        pair_q(KBits<16>{});
        attend_pages<D, VB, false, 16>(kl, vl, T % BLOCK, kl, vl, 0, qw, A, sl, g, c);
      }
    }
  }

  // After a wait gives up the warp takes nothing more; the copies still in
  // flight are waited for (bounded) before the CTA reuses the stage memory.
  bool ok = true;
  // (With the test hook dbg_wait_expiry set, a wait that saw its copy land still
  // reports expiry, so the timeout path runs with no copy left in flight.)
  const bool expire = st.dbg_wait_expiry != 0;
  // Wait for page j in stage si, the (q)-th copy into that stage: first until the
  // copy was issued (the stage's previous page done), then for its barrier phase.
  // Warp-uniform outcome: the MMAs that follow need every lane.
  auto wait_page = [&](int j, int si, uint32_t q) {
    bool landed = true;
    for (int i = 0; *reinterpret_cast<volatile int*>(&s_issued[si]) != j; ++i)
      if (i == WAIT_LIMIT) {
        landed = false;
        break;
      }
    landed = landed && mbar_wait(bar0 + 8 * si, q & 1u);
    if (!__all_sync(0xffffffffu, landed && !expire) && ok) {
      ok = false;
      if (lane == 0) set_error(st, EKV_ETIMEOUT);
    }
  };
  // Lanes 0 and 1 copy pages k + ns and k + 1 + ns into the stages si, si + 1 of
  // pages k and k + 1.
  auto refill = [&](int k, int si, bool two) {
    const int j = k + ns + lane;
    if (lane < (two ? 2 : 1) && j < np && ok) issue(j, si + lane);
  };
  // The first page of this warp's next pair (np once there are none left).
  int next_static = 2 * warp;
  auto take = [&]() {
    int k = np;
    if (stat) {
      if (ok) k = next_static;
      next_static += 2 * NW;
      return k;
    }
    if (lane == 0 && ok) k = atomicAdd(&s_next, 2);
    return __shfl_sync(0xffffffffu, k, 0);
  };
  if (uniform) {
    // Every pipelined page of this split has format fmt_u: one K width, one
    // stage layout, no per-page format decode.
    with_kbits(bits_of_code(fmt_u >> 2), [&](auto kbc) {
      constexpr int KB = decltype(kbc)::value;
      constexpr int KP = k_part_bytes(KB, D, ASYM);
      pair_q(kbc);
      // One loop per assignment, chosen once (the static one waits on its own
      // stages' barriers directly: their copies were issued before its wait).
      auto loop = [&](auto stat_c) {
        constexpr bool STAT = decltype(stat_c)::value;
        for (int it = 0;; ++it) {
          int k;
          if constexpr (STAT)
            k = ok ? 2 * (warp + NW * it) : np;
          else
            k = take();
          if (k >= np) break;
          const bool two = k + 1 < np;
          const uint32_t q = __umulhi((uint32_t)k, ns_magic);  // k even, ns even: k+1 in si+1
          const int si = k - (int)q * ns;
          if constexpr (STAT) {  // pair barrier (a uniform split with static assignment)
            const bool l0 = mbar_wait(bar0 + 8 * (si >> 1), q & 1u);
            if (!__all_sync(0xffffffffu, l0 && !expire) && ok) {
              ok = false;
              if (lane == 0) set_error(st, EKV_ETIMEOUT);
            }
            // The stages of this warp's previous pair (k - 2 NW, read before the
            // wait's vote) are refilled here rather than right after their
            // computation: the copy instructions then follow a wait instead of
            // the loads and MMAs still in flight (0.6 us less per 70B launch).
            // The warp's last pair needs no refill (its page + ns >= np).
            if (it > 0) {
              const int kp = k - 2 * NW;
              refill(kp, kp - (int)__umulhi((uint32_t)kp, ns_magic) * ns, true);
            }
          } else {
            wait_page(k, si, q);
            if (two) wait_page(k + 1, si + 1, q);
          }
          const uint8_t* sa = smem + si * stage_bytes;
          const uint8_t* sb = sa + stage_bytes;
          if (ok) {
            if (two)
              attend_pages<D, VB, true, KB>(SLd{sa}, SLd{sa + KP}, BLOCK, SLd{sb},
                                            SLd{sb + KP}, BLOCK, qw, A, sl, g, c);
            else
              attend_pages<D, VB, true, KB>(SLd{sa}, SLd{sa + KP}, BLOCK, SLd{sa}, SLd{sa}, 0,
                                            qw, A, sl, g, c);
          }
          if constexpr (!STAT) {
            __syncwarp();
            refill(k, si, two);
          }
        }
      };
      if (stat)
        loop(BoolC<true>{});
      else
        loop(BoolC<false>{});
    });
  } else {
    while (true) {
      const int k = take();
      if (k >= np) break;
      const bool two = k + 1 < np;
      const uint32_t q = __umulhi((uint32_t)k, ns_magic);
      const int si = k - (int)q * ns;
      const int32_t ea = s_bt[k];
      const int32_t eb = two ? s_bt[k + 1] : -1;
      if (ea != -1) wait_page(k, si, q);
      if (eb != -1) wait_page(k + 1, si + 1, q);
      const uint8_t* sa = smem + si * stage_bytes;
      const uint8_t* sb = sa + stage_bytes;
      const int kba = ea != -1 && ok ? bits_of_code(entry_fmt(ea) >> 2) : 0;
      const int kbb = eb != -1 && ok ? bits_of_code(entry_fmt(eb) >> 2) : 0;
      if (kba != 0 && kba == kbb) {  // both pages share a K width
        with_kbits(kba, [&](auto kbc) {
          constexpr int KB = decltype(kbc)::value;
          constexpr int KP = k_part_bytes(KB, D, ASYM);
          pair_q(kbc);
          attend_pages<D, VB, true, KB>(SLd{sa}, SLd{sa + KP}, BLOCK, SLd{sb}, SLd{sb + KP},
                                        BLOCK, qw, A, sl, g, c);
        });
      } else {  // one page at a time, through one call site per K width
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          const int kbx = pass ? kbb : kba;
          if (kbx == 0) continue;
          const uint8_t* x = pass ? sb : sa;
          with_kbits(kbx, [&](auto kbc) {
            constexpr int KB = decltype(kbc)::value;
            pair_q(kbc);
            attend_pages<D, VB, true, KB>(SLd{x}, SLd{x + k_part_bytes(KB, D, ASYM)}, BLOCK,
                                          SLd{x}, SLd{x}, 0, qw, A, sl, g, c);
          });
        }
      }
      __syncwarp();
      refill(k, si, two);
    }
  }
  // Copies still in flight (pages no warp took after a wait gave up) land before
  // the stage memory is reused: each stage waits, bounded, for its last copy.
  __syncthreads();
  // (With pair barriers only the even stage of a pair is checked: it holds the
  // pair's latest page, and the odd stage's may be a round older.)
  if (tid < ns && !(pairb && (tid & 1)) && s_issued[tid] >= 0 &&
      !mbar_wait(bar0 + 8 * (pairb ? tid >> 1 : tid),
                 __umulhi((uint32_t)s_issued[tid], ns_magic) & 1u))
    set_error(st, EKV_ETIMEOUT);
  __syncthreads();  // every stage drained before the stage memory is reused

  // ---- remove the V code bias: o_c = (o_c - vbias(c) * sum P') / vmul(c) ------------
  // Channel c of m-tile mt, rows g and g+8, has chunk index mt or NMT + mt, whose
  // class (position of its code in the word) depends on mt only.
  if constexpr (vbias_trick<VB>()) {
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      const float bias = vbias<VB>(mt), inv = 1.f / vmul<VB>(mt);
      A.o[mt][0] = (A.o[mt][0] - bias * A.ps[0]) * inv;
      A.o[mt][1] = (A.o[mt][1] - bias * A.ps[1]) * inv;
      A.o[mt][2] = (A.o[mt][2] - bias * A.ps[0]) * inv;
      A.o[mt][3] = (A.o[mt][3] - bias * A.ps[1]) * inv;
    }
  }

  if constexpr (ASYM && VB < 16) {  // + sum_t p_t z_t on every channel of the head
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      A.z0 += __shfl_xor_sync(0xffffffffu, A.z0, off);
      A.z1 += __shfl_xor_sync(0xffffffffu, A.z1, off);
    }
#pragma unroll
    for (int mt = 0; mt < NMT; ++mt) {
      A.o[mt][0] += A.z0;
      A.o[mt][1] += A.z1;
      A.o[mt][2] += A.z0;
      A.o[mt][3] += A.z1;
    }
  }

  // ---- merge the warps of this CTA (reusing the stage memory) ----------------------
  float* sm_acc = reinterpret_cast<float*>(smem);  // [NW][SLOTS]
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    A.l0 += __shfl_xor_sync(0xffffffffu, A.l0, off);
    A.l1 += __shfl_xor_sync(0xffffffffu, A.l1, off);
  }
  if (g == 0) {
    sm_m[warp][2 * c] = A.m0; sm_m[warp][2 * c + 1] = A.m1;
    sm_l[warp][2 * c] = A.l0; sm_l[warp][2 * c + 1] = A.l1;
  }
  constexpr int SLOTS = MergeShape<D, NT>::SLOTS, PTS = MergeShape<D, NT>::PTS;
  float* wacc = sm_acc + (size_t)warp * SLOTS + lane;
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
    for (int j = 0; j < 4; ++j) wacc[(mt * 4 + j) * 32] = A.o[mt][j];
  __syncthreads();
  // Per head (one warp per head, lane w holding warp w's state): the CTA's max,
  // each warp's weight 2^(m_w - M) and the weighted sum, by shuffles.
  static_assert(NW <= 32, "one lane per warp of the CTA");
  for (int hd = warp; hd < G; hd += NW) {
    const float mw = lane < NW ? sm_m[lane][hd] : -CUDART_INF_F;
    const float lw = lane < NW ? sm_l[lane][hd] : 0.f;
    float M = mw;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float f = mw == -CUDART_INF_F ? 0.f : exp2f(mw - M);
    float L = f * lw;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane < NW) sm_f[lane][hd] = f;
    if (lane == 0) {
      sm_ml[hd][0] = M;
      sm_ml[hd][1] = L;
    }
  }
  __syncthreads();

  // Launched as a programmatic dependent, everything above overlapped the end of
  // the launch before it in the stream, which may still be using the shared
  // split scratch and O: wait for it here (a no-op otherwise), then let the next
  // launch start (unless the early wait above already did).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!(PACK == 1 && dep_inputs)) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const size_t pbase = ((size_t)z * st.Hkv + h) * splits;
  const size_t pid = pbase + split;
  __half* orow = o + ((size_t)z * st.Hq + h * G) * D;
  {
    const int hd = slot_head<D>(tid);
    if (hd < G) {
      float r[PTS];
#pragma unroll
      for (int k = 0; k < PTS; ++k) r[k] = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = sm_f[w][hd];
#pragma unroll
        for (int k = 0; k < PTS; ++k)
          if (tid + k * NT < SLOTS) r[k] = fmaf(f, sm_acc[(size_t)w * SLOTS + tid + k * NT], r[k]);
      }
      if (splits == 1) {
        const float L = sm_ml[hd][1], inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int k = 0; k < PTS; ++k)
          if (tid + k * NT < SLOTS)
            orow[hd * D + slot_ch<D>(tid + k * NT)] = __float2half_rn(r[k] * inv);
      } else {
#pragma unroll
        for (int k = 0; k < PTS; ++k)
          if (tid + k * NT < SLOTS) st.attn_acc[pid * SLOTS + tid + k * NT] = r[k];
        if ((tid & ~32) < 4)
          *reinterpret_cast<float2*>(st.attn_ml + (pid * MAX_G + hd) * 2) =
              make_float2(sm_ml[hd][0], sm_ml[hd][1]);
      }
    }
  }
  // The new length is published once every CTA of the sequence has read the old
  // one: one arrival per KV head, from its only CTA or from the CTA that merges
  // its splits (all of which have arrived by then).
  auto publish_length = [&]() {
    if constexpr (FUSED) {
      if (app && tid == 0) {
        int* tk = st.append_ticket + ls_index(st, layer, slot);
        if (atomicAdd(tk, 1) == st.Hkv - 1) {
          st.len[ls_index(st, layer, slot)] = T;
          *tk = 0;
        }
      }
    }
  };
  if (splits == 1) {
    publish_length();
    return;
  }

  // ---- merge of the splits ------------------------------------------------------------
  // Up to ATTN_GROUP splits: the last CTA to finish merges them all into O.  More:
  // splits form groups of ATTN_GROUP, the last CTA of each group merges the group
  // into the slot of its first split, and the last group merger merges the groups
  // into O.  Tickets never wait.
  const int grp = split / ATTN_GROUP, ngrp = (splits + ATTN_GROUP - 1) / ATTN_GROUP;
  const int gsize = min(ATTN_GROUP, splits - grp * ATTN_GROUP);
  int* tk = st.attn_ticket + ((size_t)z * st.Hkv + h) * ATTN_TICKETS;
  if (!last_arrival(tk + 1 + grp, gsize, tid, &s_last)) return;
  if (ngrp == 1) {
    if constexpr (MergeShape<D, NT>::PTS <= 2)  // every partial's slots fit the registers
      merge_final<D, NT>(st.attn_acc, st.attn_ml, pbase, splits, G, tid, orow, sm_mf, sm_inv);
    else
      merge_parts<D, NT>(st.attn_acc, st.attn_ml, pbase, 0, 1, splits, G, tid, orow, 0);
    publish_length();
    return;
  }
  merge_parts<D, NT>(st.attn_acc, st.attn_ml, pbase, grp * ATTN_GROUP, 1, gsize, G, tid,
                     nullptr, pbase + grp * ATTN_GROUP);
  if (!last_arrival(tk, ngrp, tid, &s_last)) return;
  merge_parts<D, NT>(st.attn_acc, st.attn_ml, pbase, 0, ATTN_GROUP, ngrp, G, tid, orow, 0);
  publish_length();
}

template <int D, int VB, int PACK>
cudaError_t launch_t(const DevState& st, int layer, int n_seqs, const int32_t* slots,
                     const __half* q, __half* o, int splits, const __half* knew,
                     const __half* vnew, int overlap, cudaStream_t s) {
  using Cfg = AttnCfg<VB, PACK>;
  dim3 grid(splits * st.Hkv * n_seqs);
  if (knew && overlap) {  // programmatic dependent of the launch before it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Cfg::NT);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_attn_kernel<D, VB, true, PACK>, st, layer, slots, q,
                              o, splits, knew, vnew, ATTN_LATE_BLOCKS,
                              overlap == OVERLAP_DEPENDENT ? 1 : 0);
  }
  if (knew)
    decode_attn_kernel<D, VB, true, PACK><<<grid, Cfg::NT, Cfg::SMEM, s>>>(
        st, layer, slots, q, o, splits, knew, vnew, 0, 0);
  else
    decode_attn_kernel<D, VB, false, PACK><<<grid, Cfg::NT, Cfg::SMEM, s>>>(
        st, layer, slots, q, o, splits, nullptr, nullptr, 0, 0);
  return cudaGetLastError();
}

template <int D, int VB, int PACK>
cudaError_t init_pack() {
  cudaError_t e = cudaSuccess;
  for (auto fn : {decode_attn_kernel<D, VB, false, PACK>, decode_attn_kernel<D, VB, true, PACK>}) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               AttnCfg<VB, PACK>::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
  }
  return e;
}

// Two CTAs per SM are built for d = 128 with quantized V only (the batched
// shapes); the host never asks for them otherwise.
template <int D, int VB>
constexpr bool has_pack2() { return D == 128 && VB < 16; }

template <int D, int VB>
cudaError_t init_t(bool* pack2_ok) {
  cudaError_t e = init_pack<D, VB, 1>();
  if constexpr (has_pack2<D, VB>()) {
    if (e == cudaSuccess) e = init_pack<D, VB, 2>();
    // both kernels of the pair must fit twice on an SM, else the host keeps one
    // CTA per SM
    for (auto fn : {decode_attn_kernel<D, VB, false, 2>, decode_attn_kernel<D, VB, true, 2>}) {
      int n = 0;
      if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, AttnCfg<VB, 2>::NT,
                                                          AttnCfg<VB, 2>::SMEM);
      if (n < 2) *pack2_ok = false;
    }
  }
  return e;
}

}  // namespace

cudaError_t EKV_ATTN_FN(attn_init)(bool* pack2_ok) {
  cudaError_t e = cudaSuccess;
  cudaError_t (*fns[])(bool*) = {init_t<64, 2>,  init_t<64, 4>,  init_t<64, 8>,  init_t<64, 16>,
                                 init_t<128, 2>, init_t<128, 4>, init_t<128, 8>, init_t<128, 16>};
  for (auto f : fns)
    if (e == cudaSuccess) e = f(pack2_ok);
  return e;
}

cudaError_t EKV_ATTN_FN(launch_decode_attn)(const DevState& st, int layer, int n_seqs,
                                            const int32_t* slots, const __half* q, __half* o,
                                            int splits, int vb, int pack, cudaStream_t s,
                                            const __half* knew, const __half* vnew,
                                            int overlap) {
  using Fn = cudaError_t (*)(const DevState&, int, int, const int32_t*, const __half*, __half*,
                             int, const __half*, const __half*, int, cudaStream_t);
  const int vi = vb == 2 ? 0 : vb == 4 ? 1 : vb == 8 ? 2 : 3;
  static const Fn tab[2][4] = {
      {launch_t<64, 2, 1>, launch_t<64, 4, 1>, launch_t<64, 8, 1>, launch_t<64, 16, 1>},
      {launch_t<128, 2, 1>, launch_t<128, 4, 1>, launch_t<128, 8, 1>, launch_t<128, 16, 1>}};
  static const Fn tab2[3] = {launch_t<128, 2, 2>, launch_t<128, 4, 2>, launch_t<128, 8, 2>};
  if (pack == 2 && st.D == 128 && vi < 3)
    return tab2[vi](st, layer, n_seqs, slots, q, o, splits, knew, vnew, overlap, s);
  if (pack != 1) return cudaErrorInvalidValue;  // not built (the host never asks)
  return tab[st.D == 64 ? 0 : 1][vi](st, layer, n_seqs, slots, q, o, splits, knew, vnew,
                                     overlap, s);
}

}  // namespace ekv
