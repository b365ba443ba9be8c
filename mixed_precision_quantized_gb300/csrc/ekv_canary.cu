// ekv_canary.cu — the EchoKV canary KL and the per-layer tier controller.
//
// Canary ("EchoKV: watching a language model decide its own precision",
// "Show the math — what the canary actually computes"):
//   delta_{l,b} = KL( softmax(sigma Q W^T) || softmax(sigma Q quant_b(W)^T) ),
// b in {2, 4, 8}, summed over the keys of the FP16 ring window W and averaged
// over every query of the step.  W is the newest min(len, 64) K vectors of the
// (layer, sequence, KV head) ring, oldest first ("Do we store the whole cache
// in FP16? — No."); quant_b is the cache's symmetric quantizer applied per
// channel over consecutive 16-row groups of W starting at the oldest row.
//
// One CTA per (layer, sequence, KV head) holds W, its three quantize-dequantize
// copies and the group's queries in shared memory, computes the four logit
// sets, the log-softmaxes and the three KL sums of its G query heads, and
// writes one partial per reading.  The last CTA of a layer (atomic ticket, no
// waiting) adds the layer's partials in a fixed order and stores its mean
// readings.  One launch may cover several layers (a firing step's canary runs
// once, after every layer's append, over all of them: a layer's ring and
// queries are final then), so a launch fills the GPU instead of Hkv * n_seqs
// CTAs.
//
// Controller ("Show the math", EMA and pick; "Bidirectional adjustment"):
//   ema = first reading ? delta : (1-alpha) ema + alpha delta   (fp32, unfused)
//   tier = min{ b in {2,4,8} : ema_b < tau }, else 8.
#include <math_constants.h>

#include "ekv_internal.h"

namespace ekv {
namespace {

constexpr int CANARY_THREADS = 1024;
constexpr int NBITS = 3;

__device__ __forceinline__ int quant_code(float x, float s, int qm) {
  if (s == 0.f) return 0;
  const int q = __float2int_rn(__fdiv_rn(x, s));
  return min(max(q, -qm), qm);
}

template <int D>
__host__ __device__ constexpr size_t canary_smem_bytes() {
  return sizeof(float) * ((size_t)(1 + NBITS) * RING * (D + 1) + (size_t)MAX_G * D +
                          (size_t)2 * (1 + NBITS) * MAX_G * RING);
}

template <int D>
__global__ void __launch_bounds__(CANARY_THREADS)
canary_kernel(DevState st, int layer0, const int32_t* __restrict__ slots,
              const __half* __restrict__ qs, size_t q_layer_stride,
              float* __restrict__ delta_out, int n_seqs) {
  constexpr int P = D + 1;  // padded row
  extern __shared__ float sm[];
  float* W = sm;                             // [64][P]   fp16 window as fp32
  float* WQ = W + RING * P;                  // [3][64][P] quantize-dequantize copies
  float* Qs = WQ + NBITS * RING * P;         // [G][D]
  float* Z = Qs + MAX_G * D;                 // [2][4][G][64] half-sums, then logits
  __shared__ float s_kl[NBITS][MAX_G];
  __shared__ int s_last;

  const int h = blockIdx.x, z = blockIdx.y;
  const int layer = layer0 + blockIdx.z;
  const __half* q = qs + blockIdx.z * q_layer_stride;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = st.G;
  const int slot = slots[z];
  const bool ok = slot >= 0 && slot < st.S;
  const int T = ok ? st.len[ls_index(st, layer, slot)] : 0;
  const int n = min(T, RING);
  if (!ok && tid == 0) set_error(st, EKV_EINVAL);

  const __half* ring = st.ring + lsh_index(st, layer, ok ? slot : 0, h) * (RING * D);
  for (int i = tid; i < n * D; i += CANARY_THREADS) {
    const int j = i / D, c = i % D;
    W[j * P + c] = __half2float(ring[(size_t)((T - n + j) % RING) * D + c]);
  }
  for (int i = tid; i < G * D; i += CANARY_THREADS)
    Qs[i] = __half2float(q[((size_t)z * st.Hq + (size_t)h * G) * D + i]);
  __syncthreads();

  // quantize-dequantize: one task per (bit width, 16-row group, channel)
  const int ngr = (n + 15) / 16;
  for (int i = tid; i < NBITS * ngr * D; i += CANARY_THREADS) {
    const int bi = i / (ngr * D), gi = i / D % ngr, c = i % D;
    const int r0 = gi * 16, r1 = min(r0 + 16, n);
    if (st.asym) {  // KIVI-style: min/max scale, zero point lo, unsigned codes
      float lo = CUDART_INF_F, hi = -CUDART_INF_F;
      for (int r = r0; r < r1; ++r) {
        lo = fminf(lo, W[r * P + c]);
        hi = fmaxf(hi, W[r * P + c]);
      }
      const int L = (1 << (2 << bi)) - 1;
      const float sf = __half2float(__float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), (float)L)));
      for (int r = r0; r < r1; ++r) {
        const float x = W[r * P + c];
        const int u = sf == 0.f ? 0 : min(max(__float2int_rn(__fdiv_rn(__fsub_rn(x, lo), sf)), 0), L);
        WQ[(bi * RING + r) * P + c] = __fadd_rn(__fmul_rn((float)u, sf), lo);
      }
      continue;
    }
    float m = 0.f;
    for (int r = r0; r < r1; ++r) m = fmaxf(m, fabsf(W[r * P + c]));
    m = fminf(m, st.kclip[((size_t)layer * st.Hkv + h) * D + c]);  // the cache's own quantizer
    const int qm = (1 << ((2 << bi) - 1)) - 1;
    const float sf = __half2float(__float2half_rn(__fdiv_rn(m, (float)qm)));
    for (int r = r0; r < r1; ++r)
      WQ[(bi * RING + r) * P + c] = (float)quant_code(W[r * P + c], sf, qm) * sf;
  }
  __syncthreads();

  // logits of the reference and the three quantized copies: each task sums one
  // half of the channels of one (query head, key); the halves are then added
  constexpr int ZS = (1 + NBITS) * MAX_G * RING;
  for (int i = tid; i < 2 * G * RING; i += CANARY_THREADS) {
    const int half = i / (G * RING), hd = i / RING % G, j = i % RING;
    if (j >= n) continue;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    const float* qh = Qs + hd * D;
    for (int c = half * (D / 2); c < (half + 1) * (D / 2); ++c) {
      const float qc = qh[c];
      a0 = fmaf(qc, W[j * P + c], a0);
      a1 = fmaf(qc, WQ[(0 * RING + j) * P + c], a1);
      a2 = fmaf(qc, WQ[(1 * RING + j) * P + c], a2);
      a3 = fmaf(qc, WQ[(2 * RING + j) * P + c], a3);
    }
    float* zh = Z + half * ZS;
    zh[(0 * MAX_G + hd) * RING + j] = a0;
    zh[(1 * MAX_G + hd) * RING + j] = a1;
    zh[(2 * MAX_G + hd) * RING + j] = a2;
    zh[(3 * MAX_G + hd) * RING + j] = a3;
  }
  __syncthreads();
  for (int i = tid; i < (1 + NBITS) * G * RING; i += CANARY_THREADS) {
    const int v = i / (G * RING), hd = i / RING % G, j = i % RING;
    if (j >= n) continue;
    const int o = (v * MAX_G + hd) * RING + j;
    Z[o] = (Z[o] + Z[ZS + o]) * st.scale;
  }
  __syncthreads();

  // KL per query head: one warp per head, lanes over keys j and j+32
  for (int hd = warp; hd < G; hd += CANARY_THREADS / 32) {
    float lse[1 + NBITS];
#pragma unroll
    for (int v = 0; v <= NBITS; ++v) {
      const float* zz = Z + (v * MAX_G + hd) * RING;
      const float za = lane < n ? zz[lane] : -CUDART_INF_F;
      const float zb = lane + 32 < n ? zz[lane + 32] : -CUDART_INF_F;
      float m = fmaxf(za, zb);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float s = (lane < n ? expf(za - m) : 0.f) + (lane + 32 < n ? expf(zb - m) : 0.f);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      lse[v] = m + logf(s);
    }
    const float* z0 = Z + (0 * MAX_G + hd) * RING;
#pragma unroll
    for (int bi = 0; bi < NBITS; ++bi) {
      const float* zb = Z + ((1 + bi) * MAX_G + hd) * RING;
      float kl = 0.f;
      for (int j = lane; j < n; j += 32) {
        const float lp = z0[j] - lse[0];
        const float lq = zb[j] - lse[1 + bi];
        kl += expf(lp) * (lp - lq);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) kl += __shfl_xor_sync(0xffffffffu, kl, off);
      if (lane == 0) s_kl[bi][hd] = kl;
    }
  }
  __syncthreads();

  const int cta = z * st.Hkv + h;
  float* part = st.canary_part + (size_t)layer * st.S * st.Hkv * NBITS;
  if (tid < NBITS) {
    float s = 0.f;
    for (int hd = 0; hd < G; ++hd) s += n > 0 ? s_kl[tid][hd] : 0.f;
    part[(size_t)cta * NBITS + tid] = s;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int* tk = st.canary_ticket + layer;
    const int t = atomicAdd(tk, 1);
    s_last = (t == n_seqs * st.Hkv - 1);
    if (s_last) *tk = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < NBITS) {
    float s = 0.f;
    for (int i = 0; i < n_seqs * st.Hkv; ++i) s += __ldcg(part + (size_t)i * NBITS + tid);
    const float dl = s / (float)(n_seqs * st.Hq);
    st.delta[layer * NBITS + tid] = dl;
    if (delta_out) delta_out[blockIdx.z * NBITS + tid] = dl;
  }
}

__global__ void tier_update_kernel(DevState st, const float* __restrict__ delta,
                                   const uint8_t* __restrict__ mask, int freeze) {
  if (freeze) return;
  for (int l = threadIdx.x; l < st.L; l += blockDim.x) {
    if (mask && !mask[l]) continue;
    const float* d = delta ? delta + l * NBITS : st.delta + l * NBITS;
    float* e = st.ema + l * NBITS;
    const bool first = st.ema_valid[l] == 0;
    const float one_minus = __fsub_rn(1.0f, st.alpha);
    // Budget: tau, or tau * sqrt(L / L0) with L the mean length of the layer's
    // sequences that hold tokens ("The tau(L) scaling").
    float budget = st.tau;
    if (st.tau_ctx0 > 0) {
      long long sum = 0;
      int n = 0;
      for (int s = 0; s < st.S; ++s) {
        const int t = st.len[ls_index(st, l, s)];
        if (t > 0) {
          sum += t;
          ++n;
        }
      }
      if (n > 0) {
        const float mean = __fdiv_rn((float)sum, (float)n);
        budget = __fmul_rn(st.tau, __fsqrt_rn(__fdiv_rn(mean, (float)st.tau_ctx0)));
      }
    }
    // Fewer bits than the current tier must clear the budget by the hysteresis.
    const int cur = st.tier[l];
    const float lower = __fmul_rn(budget, __fsub_rn(1.0f, st.hyst));
    int pick = 8;
    bool picked = false;
#pragma unroll
    for (int bi = 0; bi < NBITS; ++bi) {
      const float v = first ? d[bi]
                            : __fadd_rn(__fmul_rn(one_minus, e[bi]), __fmul_rn(st.alpha, d[bi]));
      e[bi] = v;
      if (!picked && v < ((2 << bi) < cur ? lower : budget)) {
        pick = 2 << bi;
        picked = true;
      }
    }
    st.ema_valid[l] = 1;
    // A new tier needs `vote` consecutive firings that pick it.
    if (pick == cur) {
      st.cnt[l] = 0;
    } else {
      int n = st.cand[l] == pick ? st.cnt[l] + 1 : 1;
      if (n >= st.vote) {
        st.tier[l] = pick;
        n = 0;
      }
      st.cand[l] = pick;
      st.cnt[l] = n;
    }
  }
}

}  // namespace

cudaError_t canary_init() {
  cudaError_t e = cudaFuncSetAttribute(canary_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)canary_smem_bytes<64>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(canary_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)canary_smem_bytes<128>());
  return e;
}

cudaError_t launch_canary(const DevState& st, int layer0, int n_layers, int n_seqs,
                          const int32_t* slots, const __half* q, size_t q_layer_stride,
                          float* delta_out, cudaStream_t s) {
  dim3 grid(st.Hkv, n_seqs, n_layers);
  if (st.D == 64)
    canary_kernel<64><<<grid, CANARY_THREADS, canary_smem_bytes<64>(), s>>>(
        st, layer0, slots, q, q_layer_stride, delta_out, n_seqs);
  else
    canary_kernel<128><<<grid, CANARY_THREADS, canary_smem_bytes<128>(), s>>>(
        st, layer0, slots, q, q_layer_stride, delta_out, n_seqs);
  return cudaGetLastError();
}

cudaError_t launch_tier_update(const DevState& st, const float* delta, const uint8_t* mask,
                               int freeze, cudaStream_t s) {
  tier_update_kernel<<<1, 128, 0, s>>>(st, delta, mask, freeze);
  return cudaGetLastError();
}

}  // namespace ekv
