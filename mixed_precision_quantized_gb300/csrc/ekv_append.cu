// ekv_append.cu — quantize-and-append into the paged cache, plus page bookkeeping kernels.
//
// Follows "EchoKV: watching a language model decide its own precision":
//   * "How EchoKV works": every step's K goes into the layer's FP16 ring before
//     it is quantized into the paged cache, and the tier vector routes future K
//     blocks to the right pool;
//   * "What happens to old blocks when a layer changes tier?": a page keeps the
//     bit-width it was admitted with.
// and "Behavior-Guided KV-Cache Quantization", "K/V Role-Aware Low-Bit
// Quantization": K is quantized per channel (here over the 16 tokens of a
// page), V per token (over the head's channels), both symmetric.
//
// One CTA handles one (sequence, KV head, touched block).  The block's page is
// popped from the free stack of format (tier, V bits) when the block's first
// token arrives.  V rows are quantized at once; K rows wait in the block's fp16
// staging rows until the 16th token seals the block.  The CTA that finishes
// last for a sequence (atomic ticket) publishes the new length, so every CTA
// reads the old length first.
#include "ekv_internal.h"
#include "ekv_quant.cuh"

namespace ekv {
namespace {

constexpr int APPEND_THREADS = 128;

template <int D>
__global__ void __launch_bounds__(APPEND_THREADS)
append_kernel(DevState st, int layer, const int32_t* __restrict__ slots, int n_new,
              const __half* __restrict__ k, const __half* __restrict__ v) {
  constexpr int CH = D / 8;
  const int jj = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NWARP = APPEND_THREADS / 32;
  __shared__ int s_told, s_entry;

  const int slot = slots[z];
  if (slot < 0 || slot >= st.S) {
    if (tid == 0) set_error(st, EKV_EINVAL);
    return;
  }
  if (tid == 0) s_told = st.len[ls_index(st, layer, slot)];
  __syncthreads();
  const int told = s_told, tnew = told + n_new;
  if (tnew > st.maxblk * BLOCK) {  // would outgrow the block table: nothing is written
    if (tid == 0 && jj == 0 && h == 0) set_error(st, EKV_ESTATE);
    return;
  }
  const int j = told / BLOCK + jj;
  const int lo = max(j * BLOCK, told), hi = min(j * BLOCK + BLOCK, tnew);
  const size_t in_row = (size_t)st.Hkv * D;
  const __half* kin = k + (size_t)z * n_new * in_row + (size_t)h * D;
  const __half* vin = v + (size_t)z * n_new * in_row + (size_t)h * D;

  if (lo < hi) {
    if (tid == 0) {
      int32_t* btp = st.bt + lsh_index(st, layer, slot, h) * st.maxblk + j;
      int32_t e;
      if (j * BLOCK >= told) {  // block opens now: admit at the layer's current tier
        const int fmt = code_of_bits(st.tier[layer]) * 4 + code_of_bits(st.vbits[layer]);
        const int old = atomicSub(st.top + fmt, 1);
        if (old <= 0) {
          atomicAdd(st.top + fmt, 1);
          set_error(st, EKV_ENOMEM);
          e = -1;
        } else {
          e = (int32_t)(((uint32_t)fmt << 28) | (uint32_t)st.stack[fmt][old - 1]);
          atomicMax(st.kmax + layer, st.tier[layer]);
        }
        *btp = e;
      } else {
        e = *btp;
      }
      s_entry = e;
    }
    __syncthreads();
    const int32_t e = s_entry;
    __half* stg = st.staging + lsh_index(st, layer, slot, h) * (BLOCK * D);
    if (e != -1) {
      const int fmt = entry_fmt(e);
      const int kb = bits_of_code(fmt >> 2), vb = bits_of_code(fmt & 3);
      uint8_t* page = st.pool_base[fmt] + (size_t)entry_idx(e) * st.pool_page_bytes[fmt];
      uint8_t* vpart = page + k_part_bytes(kb, D, st.asym);
      const size_t lh = (size_t)layer * st.Hkv + h;
      const float vc = st.vclip[lh];
      for (int p = lo + warp; p < hi; p += NWARP) {
        const __half* src = vin + (size_t)(p - told) * in_row;
        if (st.asym) quant_v_row<D, true>(src, vpart, p - j * BLOCK, vb, lane, vc);
        else quant_v_row<D, false>(src, vpart, p - j * BLOCK, vb, lane, vc);
      }
      if (hi == j * BLOCK + BLOCK) {
        if (tid < CH) {
          if (st.asym) seal_k<D, true>(stg, kin, in_row, j, told, kb, page, tid, st.kclip + lh * D);
          else seal_k<D, false>(stg, kin, in_row, j, told, kb, page, tid, st.kclip + lh * D);
        }
      } else {
        for (int i = tid; i < (hi - lo) * CH; i += APPEND_THREADS) {
          const int p = lo + i / CH, cc = i % CH;
          *reinterpret_cast<uint4*>(stg + (size_t)(p - j * BLOCK) * D + 8 * cc) =
              *reinterpret_cast<const uint4*>(kin + (size_t)(p - told) * in_row + 8 * cc);
        }
      }
    } else if (j * BLOCK < told) {  // an existing block must have a page
      if (tid == 0) set_error(st, EKV_ESTATE);
    }
    // ring: the newest 64 K vectors, slot p % 64
    __half* ring = st.ring + lsh_index(st, layer, slot, h) * (RING * D);
    const int rlo = max(lo, tnew - RING);
    for (int i = tid; i < (hi - rlo) * CH && rlo < hi; i += APPEND_THREADS) {
      const int p = rlo + i / CH, cc = i % CH;
      *reinterpret_cast<uint4*>(ring + (size_t)(p % RING) * D + 8 * cc) =
          *reinterpret_cast<const uint4*>(kin + (size_t)(p - told) * in_row + 8 * cc);
    }
  }

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int total = gridDim.x * gridDim.y;
    int* tk = st.append_ticket + ls_index(st, layer, slot);
    if (atomicAdd(tk, 1) == total - 1) {
      st.len[ls_index(st, layer, slot)] = tnew;
      *tk = 0;
    }
  }
}

// Return every page of one sequence slot to its pool; one CTA per layer.
__global__ void seq_reset_kernel(DevState st, int slot) {
  const int l = blockIdx.x;
  const int n = st.Hkv * st.maxblk;
  int32_t* bt = st.bt + lsh_index(st, l, slot, 0) * st.maxblk;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int32_t e = bt[i];
    if (e == -1) continue;
    const int fmt = entry_fmt(e);
    const int pos = atomicAdd(st.top + fmt, 1);
    if (pos < st.pool_cap[fmt]) st.stack[fmt][pos] = entry_idx(e);
    else set_error(st, EKV_ESTATE);
    bt[i] = -1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    st.len[ls_index(st, l, slot)] = 0;
    st.append_ticket[ls_index(st, l, slot)] = 0;
  }
}

__global__ void read_pages_kernel(DevState st, int layer, int slot, int h, int first,
                                  uint8_t* dst, size_t stride) {
  const int i = blockIdx.x, j = first + i;
  if (j >= st.maxblk) return;
  const int32_t e = st.bt[lsh_index(st, layer, slot, h) * st.maxblk + j];
  if (e == -1) return;
  const int fmt = entry_fmt(e);
  const uint8_t* page = st.pool_base[fmt] + (size_t)entry_idx(e) * st.pool_page_bytes[fmt];
  const int n16 = st.pool_page_bytes[fmt] / 16;
  for (int c = threadIdx.x; c < n16; c += blockDim.x)
    reinterpret_cast<uint4*>(dst + (size_t)i * stride)[c] = reinterpret_cast<const uint4*>(page)[c];
}

// Page census of layers l0 .. l0 + gridDim.x / S - 1: one CTA per (layer, slot).
// cnt (dev uint64 [3 * NFMT + 1], zeroed by the caller): sealed pages per format,
// open pages per format (a sequence's last block while it holds under 16
// tokens), the tokens of those open blocks per format, and blocks in use
// without a page.
__global__ void stats_kernel(DevState st, int l0, unsigned long long* cnt) {
  __shared__ unsigned long long sc[3 * NFMT + 1];
  const int l = l0 + blockIdx.x / st.S, s = blockIdx.x % st.S;
  for (int i = threadIdx.x; i <= 3 * NFMT; i += blockDim.x) sc[i] = 0;
  __syncthreads();
  const int T = st.len[ls_index(st, l, s)];
  const int nb = (T + BLOCK - 1) / BLOCK, open = T % BLOCK;
  for (int i = threadIdx.x; i < st.Hkv * nb; i += blockDim.x) {
    const int h = i / nb, j = i % nb;
    const int32_t e = st.bt[lsh_index(st, l, s, h) * st.maxblk + j];
    if (e == -1) {  // a block in use must have a page
      atomicAdd(&sc[3 * NFMT], 1ull);
      continue;
    }
    const int f = entry_fmt(e);
    if (open && j == nb - 1) {
      atomicAdd(&sc[NFMT + f], 1ull);
      atomicAdd(&sc[2 * NFMT + f], (unsigned long long)open);
    } else {
      atomicAdd(&sc[f], 1ull);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= 3 * NFMT; i += blockDim.x)
    if (sc[i]) atomicAdd(cnt + i, sc[i]);
}

__global__ void init_stack_kernel(int32_t* stack, int32_t n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    stack[i] = i;
}

}  // namespace

cudaError_t launch_append(const DevState& st, int layer, int n_seqs, const int32_t* slots,
                          int n_new, const __half* k, const __half* v, cudaStream_t s) {
  // blocks touched by n_new tokens starting anywhere inside a block
  const int nt = (n_new + BLOCK - 2) / BLOCK + 1;
  dim3 grid(nt, st.Hkv, n_seqs);
  if (st.D == 64)
    append_kernel<64><<<grid, APPEND_THREADS, 0, s>>>(st, layer, slots, n_new, k, v);
  else
    append_kernel<128><<<grid, APPEND_THREADS, 0, s>>>(st, layer, slots, n_new, k, v);
  return cudaGetLastError();
}

cudaError_t launch_seq_reset(const DevState& st, int slot, cudaStream_t s) {
  seq_reset_kernel<<<st.L, 256, 0, s>>>(st, slot);
  return cudaGetLastError();
}

cudaError_t launch_read_pages(const DevState& st, int layer, int slot, int h, int first, int n,
                              uint8_t* dst, size_t stride, cudaStream_t s) {
  read_pages_kernel<<<n, 128, 0, s>>>(st, layer, slot, h, first, dst, stride);
  return cudaGetLastError();
}

cudaError_t launch_stats(const DevState& st, int l0, int nl, unsigned long long* cnt,
                         cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(cnt, 0, (3 * NFMT + 1) * sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  stats_kernel<<<nl * st.S, 256, 0, s>>>(st, l0, cnt);
  return cudaGetLastError();
}

cudaError_t launch_init_stack(int32_t* stack, int32_t n, cudaStream_t s) {
  const int blocks = (int)min((n + 255) / 256, 4096);
  init_stack_kernel<<<blocks > 0 ? blocks : 1, 256, 0, s>>>(stack, n);
  return cudaGetLastError();
}

}  // namespace ekv
