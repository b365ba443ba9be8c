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
// group's own values.  Each pass splits the rows over about four waves of
// CTAs; a CTA counts in shared memory and adds its counts to a global
// histogram (caller scratch), and one thread per group then walks the bins.
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
constexpr int SEL_BINS = 256;  // first pass (key bits 14..7); the second uses 128 (bits 6..0)
constexpr int SEL_UNROLL = 32;  // rows in flight per warp (column groups)
constexpr int SEL_RU = 4;       // rows in flight per warp (segment groups)

__device__ __forceinline__ uint32_t mag_key(__half x) { return __half_as_ushort(x) & 0x7fffu; }

// Histogram of one pass over one row chunk, added to the global histogram
// G[group][bins].  Pass 0 counts key >> 7; pass 1 counts key & 127 of the keys
// whose key >> 7 equals the group's first-pass bin b1[group].
//
// COLS (group_width == 1): CTA = 32 consecutive groups x one row chunk; warp w
// takes rows w, w+8, ...; lane i owns group g0+i, so a warp reads 32
// neighbouring elements of one row (64 contiguous bytes when group_stride == 1)
// and each lane writes only its own group's histogram row.
// Segments (group_width > 1): CTA = one group x one row chunk; lanes read along
// the segment, warps take rows; per-warp histograms keep shared-memory atomics
// off one hot row.
template <bool COLS>
__global__ void __launch_bounds__(SEL_THREADS)
select_hist_kernel(const __half* __restrict__ x, int64_t n_rows, int64_t row_stride,
                   int n_groups, int64_t group_stride, int width, int64_t rows_per_cta, int pass,
                   const int32_t* __restrict__ b1, uint32_t* __restrict__ G) {
  constexpr int NH = COLS ? SEL_TILE : SEL_WARPS;
  __shared__ uint32_t hist[NH][SEL_BINS + 1];  // padded: 32 lanes on one bin hit 32 banks
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nbins = pass ? 128 : SEL_BINS;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_cta;
  const int64_t r1 = min(n_rows, r0 + rows_per_cta);
  for (int i = tid; i < NH * (SEL_BINS + 1); i += SEL_THREADS) (&hist[0][0])[i] = 0;
  __syncthreads();
  if (COLS) {
    const int g = blockIdx.x * SEL_TILE + lane;
    if (g < n_groups) {
      const __half* col = x + (int64_t)g * group_stride;
      const uint32_t want = pass ? (uint32_t)b1[g] : 0u;
      uint32_t* h = hist[lane];
      int64_t r = r0 + warp;
      for (; r + (SEL_UNROLL - 1) * SEL_WARPS < r1; r += SEL_UNROLL * SEL_WARPS) {
        uint32_t k[SEL_UNROLL];
#pragma unroll
        for (int u = 0; u < SEL_UNROLL; ++u) k[u] = mag_key(col[(r + u * SEL_WARPS) * row_stride]);
#pragma unroll
        for (int u = 0; u < SEL_UNROLL; ++u) {
          if (!pass) atomicAdd(h + (k[u] >> 7), 1u);
          else if ((k[u] >> 7) == want) atomicAdd(h + (k[u] & 127u), 1u);
        }
      }
      for (; r < r1; r += SEL_WARPS) {
        const uint32_t k = mag_key(col[r * row_stride]);
        if (!pass) atomicAdd(h + (k >> 7), 1u);
        else if ((k >> 7) == want) atomicAdd(h + (k & 127u), 1u);
      }
    }
    __syncthreads();
    for (int i = tid; i < SEL_TILE * nbins; i += SEL_THREADS) {
      const int gi = i / nbins, b = i % nbins, g = blockIdx.x * SEL_TILE + gi;
      const uint32_t c = hist[gi][b];
      if (c && g < n_groups) atomicAdd(G + (size_t)g * SEL_BINS + b, c);
    }
  } else {
    const int g = blockIdx.x;
    const __half* base = x + (int64_t)g * group_stride;
    const uint32_t want = pass ? (uint32_t)b1[g] : 0u;
    uint32_t* h = hist[warp];
    for (int64_t r = r0 + warp; r < r1; r += SEL_RU * SEL_WARPS) {
      for (int i = lane; i < width; i += 32) {
        uint32_t k[SEL_RU];
#pragma unroll
        for (int u = 0; u < SEL_RU; ++u) {
          const int64_t ru = r + u * SEL_WARPS;
          k[u] = ru < r1 ? mag_key(base[ru * row_stride + i]) : 0xFFFFu;  // 0xFFFF: no row
        }
#pragma unroll
        for (int u = 0; u < SEL_RU; ++u) {
          if (k[u] == 0xFFFFu) continue;
          if (!pass) atomicAdd(h + (k[u] >> 7), 1u);
          else if ((k[u] >> 7) == want) atomicAdd(h + (k[u] & 127u), 1u);
        }
      }
    }
    __syncthreads();
    for (int b = tid; b < nbins; b += SEL_THREADS) {
      uint32_t c = 0;
#pragma unroll
      for (int w = 0; w < SEL_WARPS; ++w) c += hist[w][b];
      if (c) atomicAdd(G + (size_t)g * SEL_BINS + b, c);
    }
  }
}

// One thread per group: the smallest bin whose inclusive prefix count reaches
// the rank.  Pass 0 keeps that bin and the rank left inside it (and clears the
// group's histogram for pass 1); pass 1 assembles the key and writes the value.
__global__ void select_pick_kernel(uint32_t* __restrict__ G, int n_groups, int pass,
                                   uint32_t rank, int32_t* __restrict__ b1,
                                   uint32_t* __restrict__ rem, float* __restrict__ out) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n_groups) return;
  uint32_t* h = G + (size_t)g * SEL_BINS;
  const int nbins = pass ? 128 : SEL_BINS;
  const uint32_t r = pass ? rem[g] : rank;
  uint32_t acc = 0;
  int bin = nbins - 1;
  uint32_t left = 1;
  for (int b = 0; b < nbins; ++b) {
    if (acc + h[b] >= r) {
      bin = b;
      left = r - acc;
      break;
    }
    acc += h[b];
  }
  if (pass == 0) {
    b1[g] = bin;
    rem[g] = left;
    for (int b = 0; b < SEL_BINS; ++b) h[b] = 0;
  } else {
    out[g] = __half2float(__ushort_as_half((unsigned short)(((uint32_t)b1[g] << 7) | bin)));
  }
}

// Sums of (a - b)^2 and b^2 over n fp16 elements, in fp64: a grid-stride loop,
// a warp reduction and one atomic add per warp into acc[2] (zeroed by the caller).
__global__ void __launch_bounds__(256) output_error_kernel(const __half* __restrict__ a,
                                                           const __half* __restrict__ b, int64_t n,
                                                           double* __restrict__ acc) {
  double e = 0.0, r = 0.0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const double y = (double)__half2float(b[i]);
    const double d = (double)__half2float(a[i]) - y;
    e = fma(d, d, e);
    r = fma(y, y, r);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    e += __shfl_xor_sync(0xffffffffu, e, off);
    r += __shfl_xor_sync(0xffffffffu, r, off);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(acc, e);
    atomicAdd(acc + 1, r);
  }
}

}  // namespace

size_t abs_percentile_scratch_bytes(int n_groups) {
  return (size_t)n_groups * (SEL_BINS + 2) * 4;
}

cudaError_t launch_abs_percentile(const __half* x, int64_t n_rows, int64_t row_stride,
                                  int n_groups, int64_t group_stride, int width, uint32_t rank,
                                  float* out, void* scratch, int num_sm, cudaStream_t s) {
  uint32_t* G = static_cast<uint32_t*>(scratch);
  int32_t* b1 = reinterpret_cast<int32_t*>(G + (size_t)n_groups * SEL_BINS);
  uint32_t* rem = reinterpret_cast<uint32_t*>(b1 + n_groups);
  const bool cols = width == 1;
  const int64_t units = cols ? (n_groups + SEL_TILE - 1) / SEL_TILE : n_groups;
  // about four waves of CTAs, at least 64 rows each (a chunk's histogram flush
  // costs about as much as reading 64 rows)
  const int64_t want = std::max<int64_t>(1, (int64_t)4 * num_sm / units);
  const int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(
      {want, (n_rows + 63) / 64, 65535}));
  const int64_t per = (n_rows + chunks - 1) / chunks;
  const dim3 grid((unsigned)units, (unsigned)((n_rows + per - 1) / per));
  cudaError_t e = cudaMemsetAsync(G, 0, (size_t)n_groups * SEL_BINS * 4, s);
  for (int pass = 0; pass < 2 && e == cudaSuccess; ++pass) {
    if (cols)
      select_hist_kernel<true><<<grid, SEL_THREADS, 0, s>>>(x, n_rows, row_stride, n_groups,
                                                            group_stride, width, per, pass, b1, G);
    else
      select_hist_kernel<false><<<grid, SEL_THREADS, 0, s>>>(x, n_rows, row_stride, n_groups,
                                                             group_stride, width, per, pass, b1, G);
    select_pick_kernel<<<(n_groups + 127) / 128, 128, 0, s>>>(G, n_groups, pass, rank, b1, rem, out);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace ekv

using namespace ekv;

extern "C" {

int ekv_abs_percentile_scratch_bytes(int32_t n_groups, int64_t* out) {
  if (n_groups < 1 || !out) return EKV_EINVAL;
  *out = (int64_t)abs_percentile_scratch_bytes(n_groups);
  return EKV_OK;
}

int ekv_abs_percentile(const void* x, int64_t n_rows, int64_t row_stride, int32_t n_groups,
                       int64_t group_stride, int32_t group_width, double q, float* out,
                       void* scratch, int64_t scratch_bytes, void* stream) {
  if (!x || !out || !scratch || n_rows < 1 || n_groups < 1 || group_width < 1 ||
      row_stride < 0 || group_stride < 0 || !(q >= 0.0 && q <= 1.0))
    return EKV_EINVAL;
  const int64_t n = n_rows * (int64_t)group_width;
  if (n_rows > (int64_t)1 << 31 || n >= (int64_t)1 << 32) return EKV_EINVAL;  // uint32 counts
  if ((reinterpret_cast<uintptr_t>(x) & 1) || (reinterpret_cast<uintptr_t>(out) & 3) ||
      (reinterpret_cast<uintptr_t>(scratch) & 3) ||
      scratch_bytes < (int64_t)abs_percentile_scratch_bytes(n_groups))
    return EKV_EINVAL;
  int64_t r = (int64_t)std::ceil(q * (double)n);
  r = std::min<int64_t>(std::max<int64_t>(r, 1), n);
  int dev = 0, num_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return EKV_ECUDA;
  return launch_abs_percentile(static_cast<const __half*>(x), n_rows, row_stride, n_groups,
                               group_stride, group_width, (uint32_t)r, out, scratch, num_sm,
                               static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? EKV_OK
             : EKV_ECUDA;
}

int ekv_output_error(const void* o_hat, const void* o_ref, int64_t n, double* out,
                     void* scratch, void* stream) {
  if (!out || !scratch || n < 0 || (n > 0 && (!o_hat || !o_ref)) ||
      ((reinterpret_cast<uintptr_t>(o_hat) | reinterpret_cast<uintptr_t>(o_ref)) & 1) ||
      (reinterpret_cast<uintptr_t>(scratch) & 7))
    return EKV_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  double* acc = static_cast<double*>(scratch);
  int dev = 0, num_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return EKV_ECUDA;
  cudaError_t e = cudaMemsetAsync(acc, 0, 2 * sizeof(double), s);
  if (e == cudaSuccess && n > 0) {
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 4 * (int64_t)num_sm);
    output_error_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const __half*>(o_hat),
                                                          static_cast<const __half*>(o_ref), n,
                                                          acc);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpyAsync(out, acc, 2 * sizeof(double), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? EKV_OK : EKV_ECUDA;
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
