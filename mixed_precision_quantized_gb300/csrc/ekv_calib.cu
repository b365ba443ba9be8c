// ekv_calib.cu — the offline side of the static-artifact mode: percentile
// clipping thresholds from calibration tensors (a GPU radix select) and the
// AutoK layer allocator (host).
//
// "Behavior-Guided KV-Cache Quantization", "Calibration protocol" and "K/V
// Role-Aware Low-Bit Quantization": percentile candidates for the clipping
// thresholds are computed on a calibration set and frozen; "Sensitivity-Driven
// Budget Allocation": AutoK protects the fewest layers whose sensitivities reach
// a given fraction of the total.
//
// Threshold of a group = the nearest-rank quantile of |x| over its elements:
// the value of 1-based rank r (ascending) among the group's n magnitudes.  An
// fp16 magnitude orders like its 15-bit pattern (sign cleared), so the select
// runs on integer keys in two passes: a 256-bin histogram of the key's high 8
// bits finds the bin that holds rank r, a 128-bin histogram of the low 7 bits
// of the keys in that bin finds the key.  Exact: the result is one of the
// group's own values.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "ekv_internal.h"

namespace ekv {
namespace {

constexpr int SEL_THREADS = 256;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_TILE = 32;   // groups per CTA when each row holds one element of a group
constexpr int SEL_BINS = 256;  // first pass; the second uses 128

__device__ __forceinline__ uint32_t mag_key(__half x) { return __half_as_ushort(x) & 0x7fffu; }

// Smallest bin whose inclusive prefix count reaches r; returns it and the rank
// left inside it.  Sequential over the bins (one thread per group).
__device__ __forceinline__ int find_bin(const uint32_t* h, int nbins, uint32_t r, uint32_t* rem) {
  uint32_t acc = 0;
  for (int b = 0; b < nbins; ++b) {
    if (acc + h[b] >= r) {
      *rem = r - acc;
      return b;
    }
    acc += h[b];
  }
  *rem = 1;  // not reached when r <= n
  return nbins - 1;
}

// Column mode (group_width == 1): CTA = 32 consecutive groups; warp w reads
// rows w, w+8, ...; lane i owns group g0+i, so a warp reads 32 neighbouring
// elements of one row (64 contiguous bytes when group_stride == 1).  Each lane
// writes only its own group's histogram row: no two lanes of a warp collide.
__global__ void __launch_bounds__(SEL_THREADS)
select_columns_kernel(const __half* __restrict__ x, int64_t n_rows, int64_t row_stride,
                      int n_groups, int64_t group_stride, uint32_t rank, float* __restrict__ out) {
  __shared__ uint32_t hist[SEL_TILE][SEL_BINS + 1];  // padded: lanes on one bin hit 32 banks
  __shared__ int s_b1[SEL_TILE];
  __shared__ uint32_t s_rem[SEL_TILE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.x * SEL_TILE + lane;
  const bool live = g < n_groups;
  const __half* col = x + (live ? (int64_t)g * group_stride : 0);

  for (int i = tid; i < SEL_TILE * (SEL_BINS + 1); i += SEL_THREADS) (&hist[0][0])[i] = 0;
  __syncthreads();
  if (live)
    for (int64_t r = warp; r < n_rows; r += SEL_WARPS)
      atomicAdd(&hist[lane][mag_key(col[r * row_stride]) >> 7], 1u);
  __syncthreads();
  if (tid < SEL_TILE) s_b1[tid] = find_bin(hist[tid], SEL_BINS, rank, &s_rem[tid]);
  __syncthreads();
  for (int i = tid; i < SEL_TILE * (SEL_BINS + 1); i += SEL_THREADS) (&hist[0][0])[i] = 0;
  __syncthreads();
  if (live) {
    const uint32_t b1 = (uint32_t)s_b1[lane];
    for (int64_t r = warp; r < n_rows; r += SEL_WARPS) {
      const uint32_t k = mag_key(col[r * row_stride]);
      if ((k >> 7) == b1) atomicAdd(&hist[lane][k & 127u], 1u);
    }
  }
  __syncthreads();
  if (tid < SEL_TILE && blockIdx.x * SEL_TILE + tid < n_groups) {
    uint32_t rem2;
    const int b2 = find_bin(hist[tid], 128, s_rem[tid], &rem2);
    out[blockIdx.x * SEL_TILE + tid] =
        __half2float(__ushort_as_half((unsigned short)(((uint32_t)s_b1[tid] << 7) | b2)));
  }
}

// Row-segment mode (group_width > 1): CTA = one group of n_rows segments of
// group_width contiguous elements; lanes read along the segment, warps take
// rows.  Per-warp histograms keep shared-memory atomics off one hot row.
__global__ void __launch_bounds__(SEL_THREADS)
select_segments_kernel(const __half* __restrict__ x, int64_t n_rows, int64_t row_stride,
                       int64_t group_stride, int width, uint32_t rank, float* __restrict__ out) {
  __shared__ uint32_t hist[SEL_WARPS][SEL_BINS];
  __shared__ uint32_t tot[SEL_BINS];
  __shared__ int s_b1;
  __shared__ uint32_t s_rem;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const __half* base = x + (int64_t)blockIdx.x * group_stride;

  for (int pass = 0; pass < 2; ++pass) {
    for (int i = tid; i < SEL_WARPS * SEL_BINS; i += SEL_THREADS) (&hist[0][0])[i] = 0;
    __syncthreads();
    const uint32_t b1 = pass ? (uint32_t)s_b1 : 0u;
    for (int64_t r = warp; r < n_rows; r += SEL_WARPS) {
      const __half* row = base + r * row_stride;
      for (int i = lane; i < width; i += 32) {
        const uint32_t k = mag_key(row[i]);
        if (pass == 0) atomicAdd(&hist[warp][k >> 7], 1u);
        else if ((k >> 7) == b1) atomicAdd(&hist[warp][k & 127u], 1u);
      }
    }
    __syncthreads();
    for (int b = tid; b < SEL_BINS; b += SEL_THREADS) {
      uint32_t s = 0;
#pragma unroll
      for (int w = 0; w < SEL_WARPS; ++w) s += hist[w][b];
      tot[b] = s;
    }
    __syncthreads();
    if (tid == 0) {
      if (pass == 0) {
        s_b1 = find_bin(tot, SEL_BINS, rank, &s_rem);
      } else {
        uint32_t rem2;
        const int b2 = find_bin(tot, 128, s_rem, &rem2);
        out[blockIdx.x] =
            __half2float(__ushort_as_half((unsigned short)(((uint32_t)s_b1 << 7) | b2)));
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_abs_percentile(const __half* x, int64_t n_rows, int64_t row_stride,
                                  int n_groups, int64_t group_stride, int width, uint32_t rank,
                                  float* out, cudaStream_t s) {
  if (width == 1)
    select_columns_kernel<<<(n_groups + SEL_TILE - 1) / SEL_TILE, SEL_THREADS, 0, s>>>(
        x, n_rows, row_stride, n_groups, group_stride, rank, out);
  else
    select_segments_kernel<<<n_groups, SEL_THREADS, 0, s>>>(x, n_rows, row_stride, group_stride,
                                                            width, rank, out);
  return cudaGetLastError();
}

}  // namespace ekv

using namespace ekv;

extern "C" {

int ekv_abs_percentile(const void* x, int64_t n_rows, int64_t row_stride, int32_t n_groups,
                       int64_t group_stride, int32_t group_width, double q, float* out,
                       void* stream) {
  if (!x || !out || n_rows < 1 || n_groups < 1 || group_width < 1 || row_stride < 0 ||
      group_stride < 0 || !(q >= 0.0 && q <= 1.0))
    return EKV_EINVAL;
  const int64_t n = n_rows * (int64_t)group_width;
  if (n_rows > (int64_t)1 << 31 || n >= (int64_t)1 << 32) return EKV_EINVAL;  // uint32 counts
  if ((reinterpret_cast<uintptr_t>(x) & 1) || (reinterpret_cast<uintptr_t>(out) & 3))
    return EKV_EINVAL;
  int64_t r = (int64_t)std::ceil(q * (double)n);
  r = std::min<int64_t>(std::max<int64_t>(r, 1), n);
  return launch_abs_percentile(static_cast<const __half*>(x), n_rows, row_stride, n_groups,
                               group_stride, group_width, (uint32_t)r, out,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? EKV_OK
             : EKV_ECUDA;
}

int ekv_autok(const double* sensitivity, int32_t n, double frac, int32_t* order_out,
              int32_t* k_out) {
  if (n < 0 || (n > 0 && !sensitivity) || !k_out || !(frac >= 0.0 && frac <= 1.0))
    return EKV_EINVAL;
  for (int i = 0; i < n; ++i)
    if (!(sensitivity[i] >= 0.0) || !std::isfinite(sensitivity[i])) return EKV_EINVAL;
  std::vector<int32_t> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return sensitivity[a] > sensitivity[b]; });
  std::vector<double> prefix(n + 1, 0.0);
  for (int i = 0; i < n; ++i) prefix[i + 1] = prefix[i] + sensitivity[order[i]];
  const double target = frac * prefix[n];
  int k = 0;
  while (k < n && prefix[k] < target) ++k;  // prefix[n] >= target since frac <= 1
  if (order_out) std::copy(order.begin(), order.end(), order_out);
  *k_out = k;
  return EKV_OK;
}

}  // extern "C"
