// ekv_internal.h — device-side state and helpers shared by the library's kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ekv.h"

namespace ekv {

constexpr int BLOCK = EKV_BLOCK_TOKENS;  // tokens per page
constexpr int RING = EKV_RING_LEN;       // K vectors per ring
constexpr int NFMT = EKV_NUM_FORMATS;
constexpr int MAX_G = 8;                  // query heads per KV head handled by one CTA
constexpr int ATTN_MAX_SPLITS = 512;      // decode-attention splits per (sequence, KV head)
constexpr int ATTN_GROUP = 32;            // splits merged together at the first level
constexpr int ATTN_BT_CAP = 4096;         // page-table entries of one split (staged in shared memory)
constexpr int ATTN_MAXGRP = ATTN_MAX_SPLITS / ATTN_GROUP;
constexpr int ATTN_TICKETS = 1 + ATTN_MAXGRP;  // merge tickets per (sequence, KV head)

__host__ __device__ inline int bits_of_code(int code) { return 2 << code; }
__host__ __device__ inline int code_of_bits(int b) {
  return b == 2 ? 0 : b == 4 ? 1 : b == 8 ? 2 : b == 16 ? 3 : -1;
}
// Page parts.  Quantized parts hold codes, then one fp16 scale per group, then
// (asymmetric quantizer only) one fp16 zero point per group.
__host__ __device__ constexpr int k_part_bytes(int kb, int d, bool asym = false) {
  return kb == 16 ? BLOCK * d * 2 : BLOCK * d * kb / 8 + 2 * d * (asym ? 2 : 1);
}
__host__ __device__ constexpr int v_part_bytes(int vb, int d, bool asym = false) {
  return vb == 16 ? BLOCK * d * 2 : BLOCK * d * vb / 8 + 2 * BLOCK * (asym ? 2 : 1);
}
__host__ __device__ constexpr int page_bytes(int kb, int vb, int d, bool asym = false) {
  return k_part_bytes(kb, d, asym) + v_part_bytes(vb, d, asym);
}

// Page entry: (format << 28) | index, -1 = none.  Formats >= 8 make the int32
// negative, so "no page" is tested as e == -1 (index < 2^28 - 1 never forms -1).
__host__ __device__ inline int entry_fmt(int32_t e) { return (int)((uint32_t)e >> 28); }
__host__ __device__ inline int entry_idx(int32_t e) { return e & 0x0FFFFFFF; }

// Everything a kernel needs, passed by value.
struct DevState {
  int L, S, Hq, Hkv, D, G, maxblk;
  float scale;       // softmax scale sigma
  float scale_log2;  // sigma * log2(e)
  float alpha, tau;
  int tau_ctx0;      // > 0: budget scales with sqrt(mean length / tau_ctx0)
  float hyst;        // demotion margin
  int vote;          // consecutive firings a new tier needs (>= 1)
  int asym;          // 1: KIVI-style asymmetric quantizer (pages and canary)
  uint8_t* pool_base[NFMT];
  int32_t pool_page_bytes[NFMT];
  int32_t pool_cap[NFMT];
  int32_t* stack[NFMT];     // free page indices
  int32_t* top;             // [NFMT] free-stack heights
  int32_t* len;             // [L][S]
  int32_t* bt;              // [L][S][Hkv][maxblk]
  __half* staging;          // [L][S][Hkv][16][D]  open-block K rows
  __half* ring;             // [L][S][Hkv][64][D]  FP16 K_ref ring
  int32_t* tier;            // [L] current K tier (bits)
  int32_t* kmax;            // [L] widest K bits any page of the layer was admitted with
  int32_t* vbits;           // [L]
  float* ema;               // [L][3]
  int32_t* ema_valid;       // [L]
  int32_t* cand;            // [L] tier the last firings picked (vote)
  int32_t* cnt;             // [L] consecutive firings that picked `cand`
  float* delta;             // [L][3] last canary readings
  float* kclip;             // [L][Hkv][D] K clipping thresholds (+inf: none)
  float* vclip;             // [L][Hkv]    V clipping thresholds (+inf: none)
  int32_t* err;             // device error word
  int32_t* append_ticket;   // [L][S]
  float* attn_acc;          // [parts][G][D]   split partial numerators
  float* attn_ml;           // [parts][G][2]   split partial (max, sum), log2 domain
  int32_t* attn_ticket;     // [S][Hkv][ATTN_TICKETS] merge tickets (head, then groups)
  int32_t attn_parts_cap;
  float* canary_part;       // [L][S*Hkv][3]
  int32_t* canary_ticket;   // [L]
  int dbg_wait_expiry;      // test hook: bounded waits report expiry once their copy landed
};

__device__ inline void set_error(const DevState& st, int code) { atomicCAS(st.err, 0, code); }

__host__ __device__ inline size_t ls_index(const DevState& st, int l, int s) {
  return (size_t)l * st.S + s;
}
__host__ __device__ inline size_t lsh_index(const DevState& st, int l, int s, int h) {
  return ((size_t)l * st.S + s) * st.Hkv + h;
}

// ---- launchers (defined in the kernel translation units) ----------------------
cudaError_t launch_append(const DevState& st, int layer, int n_seqs, const int32_t* slots,
                          int n_new, const __half* k, const __half* v, cudaStream_t s);
cudaError_t attn_init();   // once per process, before any launch
cudaError_t attn_init_sym(bool* pack2_ok);
cudaError_t attn_init_asym(bool* pack2_ok);
bool attn_pack2_ok();      // two half-size attention CTAs fit on an SM
int attn_ctas_per_sm(int vb);  // resident decode-attention CTAs per SM for V width vb
// With knew/vnew set ([n_seqs][Hkv][d] fp16 each) the launch first appends that
// one token to every sequence (the fused decode step), then attends over it too.
// `overlap` (fused step only) launches it as a programmatic dependent of the
// stream's previous launch: OVERLAP_INDEPENDENT when that launch is the fused
// step of another layer and writes none of this call's inputs (the launch waits
// only before its writes), OVERLAP_DEPENDENT when it may write q, k and v (the
// launch reads only this layer's cache state and the slot list before it waits).
// `pack`: CTAs per SM (1, or 2 for launches with more units than SMs; see
// attn_pack in the host).
constexpr int OVERLAP_NONE = 0, OVERLAP_INDEPENDENT = 1, OVERLAP_DEPENDENT = 2;
cudaError_t launch_decode_attn(const DevState& st, int layer, int n_seqs, const int32_t* slots,
                               const __half* q, __half* o, int splits, int vb, int pack,
                               cudaStream_t s, const __half* knew = nullptr,
                               const __half* vnew = nullptr, int overlap = OVERLAP_NONE);
// The two page variants behind launch_decode_attn (st.asym picks one).
cudaError_t launch_decode_attn_sym(const DevState& st, int layer, int n_seqs,
                                   const int32_t* slots, const __half* q, __half* o, int splits,
                                   int vb, int pack, cudaStream_t s, const __half* knew,
                                   const __half* vnew, int overlap);
cudaError_t launch_decode_attn_asym(const DevState& st, int layer, int n_seqs,
                                    const int32_t* slots, const __half* q, __half* o, int splits,
                                    int vb, int pack, cudaStream_t s, const __half* knew,
                                    const __half* vnew, int overlap);
cudaError_t canary_init();  // once per process, before any launch
// Layers layer0 .. layer0+n_layers-1 in one launch; layer layer0+i reads its
// queries at q + i * q_layer_stride and writes delta_out[i][3] (if not null).
cudaError_t launch_canary(const DevState& st, int layer0, int n_layers, int n_seqs,
                          const int32_t* slots, const __half* q, size_t q_layer_stride,
                          float* delta_out, cudaStream_t s);
cudaError_t launch_tier_update(const DevState& st, const float* delta, const uint8_t* mask,
                               int freeze, cudaStream_t s);
cudaError_t launch_seq_reset(const DevState& st, int slot, cudaStream_t s);
cudaError_t launch_read_pages(const DevState& st, int layer, int slot, int h, int first, int n,
                              uint8_t* dst, size_t stride, cudaStream_t s);
cudaError_t launch_init_stack(int32_t* stack, int32_t n, cudaStream_t s);
// Page census of layers l0 .. l0+nl-1 into cnt (dev uint64 [3 * NFMT + 1]: sealed
// pages, open pages and open-block tokens per format, then blocks in use without
// a page); zeroes cnt first.
cudaError_t launch_stats(const DevState& st, int l0, int nl, unsigned long long* cnt,
                         cudaStream_t s);

// Argument checks and launch plan of decode attention for a handle: a copy of
// its device state, the split count and the layer's V bits.
int attn_plan(ekv_cache* c, int layer, int n_seqs, DevState* st, int* splits, int* vb,
              int* pack);

}  // namespace ekv
