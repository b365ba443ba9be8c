// ekv_host.cu — the C ABI: argument checks, device memory layout, launches.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <vector>

#include "ekv_internal.h"

using namespace ekv;

struct ekv_cache {
  ekv_config cfg;
  DevState st;
  std::vector<void*> allocs;
  std::vector<int> vbits;   // host copy (fixed per layer)
  int num_sm = 0;
  unsigned long long* census = nullptr;  // dev [3 * NFMT + 1], ekv_stats scratch
};

namespace {

void* dev_alloc(ekv_cache* c, size_t bytes) {
  void* p = nullptr;
  if (bytes == 0) bytes = 16;
  if (c->cfg.dev_alloc) {
    p = c->cfg.dev_alloc(bytes, c->cfg.alloc_ctx);
  } else if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    p = nullptr;
  }
  if (p) c->allocs.push_back(p);
  if (reinterpret_cast<uintptr_t>(p) & 15) return nullptr;  // every table is read in 16-byte units
  return p;
}

void free_all(ekv_cache* c) {
  for (void* p : c->allocs) {
    if (c->cfg.dev_free) c->cfg.dev_free(p, c->cfg.alloc_ctx);
    else if (!c->cfg.dev_alloc) cudaFree(p);
  }
  c->allocs.clear();
}

// CTAs per SM of a launch: 2 (half-size CTAs) when it has more (sequence, KV
// head) units than SMs, so all of them are resident at once and a caller's
// longest-first slot list pairs long and short units on the SMs instead of
// leaving a second wave; else 1.  Built for d = 128 with quantized V.
int attn_pack(const ekv_cache* c, int n_seqs, int vb) {
  return c->st.D == 128 && vb < 16 && n_seqs * c->st.Hkv > c->num_sm && attn_pack2_ok() ? 2 : 1;
}

int attn_splits(const ekv_cache* c, int n_seqs, int vb) {
  // As many splits as fit in one wave of CTAs (a partial second wave would cost
  // a whole launch's start-up and tail again).
  const int units = n_seqs * c->st.Hkv;
  const int pack = attn_pack(c, n_seqs, vb);
  const int target = attn_ctas_per_sm(vb) * pack * c->num_sm;
  int s = target / units;
  if (s < 1) s = 1;
  // A split's page-table entries must fit the kernel's shared-memory copy (the
  // splits but the last share the blocks, hence the one extra).
  const int cap = ATTN_BT_CAP / pack;
  const int need = (c->st.maxblk + cap - 1) / cap + 1;
  if (s < need) s = need;
  if (s > ATTN_MAX_SPLITS) s = ATTN_MAX_SPLITS;
  return s;
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? EKV_OK : EKV_ECUDA; }

bool valid_bits(int b) { return b == 2 || b == 4 || b == 8 || b == 16; }

}  // namespace

namespace ekv {
int attn_plan(ekv_cache* c, int layer, int n_seqs, DevState* st, int* splits, int* vb,
              int* pack) {
  if (!c || layer < 0 || layer >= c->st.L || n_seqs < 0 || n_seqs > c->st.S) return EKV_EINVAL;
  *st = c->st;
  *vb = c->vbits[layer];
  *splits = attn_splits(c, n_seqs > 0 ? n_seqs : 1, *vb);
  *pack = attn_pack(c, n_seqs > 0 ? n_seqs : 1, *vb);
  return EKV_OK;
}
}  // namespace ekv

extern "C" {

const char* ekv_status_string(int status) {
  switch (status) {
    case EKV_OK: return "ok";
    case EKV_EINVAL: return "invalid argument";
    case EKV_ENOMEM: return "out of memory (allocation failed or a page pool ran empty)";
    case EKV_ECUDA: return "CUDA error";
    case EKV_ETIMEOUT: return "device wait timed out";
    case EKV_EUNSUPPORTED: return "unsupported configuration";
    case EKV_ESTATE: return "inconsistent cache state detected on the device";
    default: return "unknown status";
  }
}

int32_t ekv_page_bytes(int32_t k_bits, int32_t v_bits, int32_t head_dim) {
  return ekv_page_bytes_q(k_bits, v_bits, head_dim, EKV_QUANT_SYMMETRIC);
}

int32_t ekv_page_bytes_q(int32_t k_bits, int32_t v_bits, int32_t head_dim, int32_t quantizer) {
  if (!valid_bits(k_bits) || !valid_bits(v_bits) || (head_dim != 64 && head_dim != 128) ||
      (quantizer != EKV_QUANT_SYMMETRIC && quantizer != EKV_QUANT_ASYMMETRIC))
    return -1;
  return page_bytes(k_bits, v_bits, head_dim, quantizer == EKV_QUANT_ASYMMETRIC);
}

int ekv_create(const ekv_config* cfg, const uint8_t* k_bits_init, const uint8_t* v_bits,
               ekv_cache** out) {
  if (!cfg || !k_bits_init || !v_bits || !out) return EKV_EINVAL;
  *out = nullptr;
  const ekv_config& k = *cfg;
  if (k.num_layers <= 0 || k.max_seqs <= 0 || k.num_kv_heads <= 0 || k.num_q_heads <= 0 ||
      k.max_seq_len <= 0)
    return EKV_EINVAL;
  if (k.num_q_heads % k.num_kv_heads) return EKV_EINVAL;
  if (k.head_dim != 64 && k.head_dim != 128) return EKV_EUNSUPPORTED;
  if (k.num_q_heads / k.num_kv_heads > MAX_G) return EKV_EUNSUPPORTED;
  if ((k.dev_alloc == nullptr) != (k.dev_free == nullptr)) return EKV_EINVAL;
  if (!(k.ema_alpha >= 0.f && k.ema_alpha <= 1.f)) return EKV_EINVAL;
  if (k.tau_ctx0 < 0 || !(k.hysteresis >= 0.f && k.hysteresis < 1.f) || k.vote < 0)
    return EKV_EINVAL;
  if (k.quantizer != EKV_QUANT_SYMMETRIC && k.quantizer != EKV_QUANT_ASYMMETRIC)
    return EKV_EINVAL;
  for (int l = 0; l < k.num_layers; ++l)
    if (!valid_bits(k_bits_init[l]) || !valid_bits(v_bits[l])) return EKV_EINVAL;
  for (int f = 0; f < NFMT; ++f)
    if (k.pool_pages[f] < 0 || k.pool_pages[f] > 0x0FFFFFFF) return EKV_EINVAL;

  ekv_cache* c = new (std::nothrow) ekv_cache();
  if (!c) return EKV_ENOMEM;
  c->cfg = k;
  DevState& st = c->st;
  memset(&st, 0, sizeof(st));
  st.L = k.num_layers;
  st.S = k.max_seqs;
  st.Hq = k.num_q_heads;
  st.Hkv = k.num_kv_heads;
  st.D = k.head_dim;
  st.G = k.num_q_heads / k.num_kv_heads;
  st.maxblk = (k.max_seq_len + BLOCK - 1) / BLOCK;
  st.scale = k.softmax_scale > 0.f ? k.softmax_scale : 1.0f / sqrtf((float)k.head_dim);
  st.scale_log2 = st.scale * 1.4426950408889634f;
  st.alpha = k.ema_alpha;
  st.tau = k.tau;
  st.tau_ctx0 = k.tau_ctx0;
  st.hyst = k.hysteresis;
  st.vote = k.vote < 1 ? 1 : k.vote;
  st.asym = k.quantizer == EKV_QUANT_ASYMMETRIC;
  c->vbits.assign(v_bits, v_bits + k.num_layers);

  int dev = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&c->num_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return EKV_ECUDA;
  }

  // The kernels' launch attributes and the two-CTA occupancy check come first:
  // the split plan below (hence the split scratch) depends on them.
  cudaError_t e = canary_init();
  if (e == cudaSuccess) e = attn_init();
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return EKV_ECUDA;
  }

  const size_t L = st.L, S = st.S, H = st.Hkv, D = st.D, MB = st.maxblk;
  bool ok = true;
  auto A = [&](size_t bytes) -> void* {
    void* p = ok ? dev_alloc(c, bytes) : nullptr;
    if (!p) ok = false;
    return p;
  };
  for (int f = 0; f < NFMT; ++f) {
    const int kb = bits_of_code(f >> 2), vb = bits_of_code(f & 3);
    st.pool_page_bytes[f] = page_bytes(kb, vb, st.D, st.asym);
    st.pool_cap[f] = (int32_t)k.pool_pages[f];
    if (k.pool_pages[f] > 0) {
      st.pool_base[f] = (uint8_t*)A((size_t)k.pool_pages[f] * st.pool_page_bytes[f]);
      st.stack[f] = (int32_t*)A((size_t)k.pool_pages[f] * 4);
    }
  }
  st.top = (int32_t*)A(NFMT * 4);
  st.len = (int32_t*)A(L * S * 4);
  st.bt = (int32_t*)A(L * S * H * MB * 4);
  st.staging = (__half*)A(L * S * H * BLOCK * D * 2);
  st.ring = (__half*)A(L * S * H * RING * D * 2);
  st.tier = (int32_t*)A(L * 4);
  st.kmax = (int32_t*)A(L * 4);
  st.vbits = (int32_t*)A(L * 4);
  st.ema = (float*)A(L * 3 * 4);
  st.ema_valid = (int32_t*)A(L * 4);
  st.cand = (int32_t*)A(L * 4);
  st.cnt = (int32_t*)A(L * 4);
  st.delta = (float*)A(L * 3 * 4);
  st.kclip = (float*)A(L * H * D * 4);
  st.vclip = (float*)A(L * H * 4);
  st.err = (int32_t*)A(4);
  st.append_ticket = (int32_t*)A(L * S * 4);
  // Split scratch for the largest plan any launch can ask for: every batch size
  // and every V width (the plan follows the same rules as the launch).
  int parts = 0;
  for (int n = 1; n <= k.max_seqs; ++n)
    for (int vb = 2; vb <= 16; vb *= 2) {
      const int p = n * k.num_kv_heads * attn_splits(c, n, vb);
      if (p > parts) parts = p;
    }
  st.attn_parts_cap = parts;
  st.attn_acc = (float*)A((size_t)parts * MAX_G * D * 4);
  st.attn_ml = (float*)A((size_t)parts * MAX_G * 2 * 4);
  st.attn_ticket = (int32_t*)A(S * H * ATTN_TICKETS * 4);
  st.canary_part = (float*)A(L * S * H * 3 * 4);
  st.canary_ticket = (int32_t*)A(L * 4);
  c->census = (unsigned long long*)A((3 * NFMT + 1) * sizeof(unsigned long long));
  if (!ok) {
    free_all(c);
    delete c;
    return EKV_ENOMEM;
  }

  auto Z = [&](void* p, size_t bytes) {
    if (e == cudaSuccess) e = cudaMemset(p, 0, bytes);
  };
  for (int f = 0; f < NFMT; ++f)
    if (k.pool_pages[f] > 0) {
      Z(st.pool_base[f], (size_t)k.pool_pages[f] * st.pool_page_bytes[f]);
      if (e == cudaSuccess) e = launch_init_stack(st.stack[f], (int32_t)k.pool_pages[f], 0);
    }
  std::vector<int32_t> top(NFMT), tiers(L), vb(L);
  for (int f = 0; f < NFMT; ++f) top[f] = (int32_t)k.pool_pages[f];
  for (size_t l = 0; l < L; ++l) {
    tiers[l] = k_bits_init[l];
    vb[l] = v_bits[l];
  }
  if (e == cudaSuccess) e = cudaMemcpy(st.top, top.data(), NFMT * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(st.tier, tiers.data(), L * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(st.vbits, vb.data(), L * 4, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(st.bt, 0xFF, L * S * H * MB * 4);
  {
    const std::vector<float> none((size_t)L * H * D, INFINITY);
    if (e == cudaSuccess) e = cudaMemcpy(st.kclip, none.data(), L * H * D * 4, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(st.vclip, none.data(), L * H * 4, cudaMemcpyHostToDevice);
  }
  Z(st.len, L * S * 4);
  Z(st.kmax, L * 4);
  Z(st.staging, L * S * H * BLOCK * D * 2);
  Z(st.ring, L * S * H * RING * D * 2);
  Z(st.ema, L * 3 * 4);
  Z(st.ema_valid, L * 4);
  Z(st.cand, L * 4);
  Z(st.cnt, L * 4);
  Z(st.delta, L * 3 * 4);
  Z(st.err, 4);
  Z(st.append_ticket, L * S * 4);
  Z(st.attn_ticket, S * H * ATTN_TICKETS * 4);
  Z(st.canary_ticket, L * 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return EKV_ECUDA;
  }
  *out = c;
  return EKV_OK;
}

int ekv_destroy(ekv_cache* c) {
  if (!c) return EKV_OK;
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
  return EKV_OK;
}

int ekv_seq_reset(ekv_cache* c, int32_t seq_slot, void* stream) {
  if (!c || seq_slot < 0 || seq_slot >= c->st.S) return EKV_EINVAL;
  return cuda_status(launch_seq_reset(c->st, seq_slot, as_stream(stream)));
}

int ekv_append(ekv_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_slots,
               int32_t n_new, const void* k, const void* v, void* stream) {
  if (!c || layer < 0 || layer >= c->st.L || n_seqs < 0 || n_seqs > c->st.S) return EKV_EINVAL;
  if (n_seqs == 0) return EKV_OK;
  if (!seq_slots || !k || !v || n_new <= 0 || n_new > c->st.maxblk * BLOCK) return EKV_EINVAL;
  if (((uintptr_t)k | (uintptr_t)v) & 15) return EKV_EINVAL;
  return cuda_status(launch_append(c->st, layer, n_seqs, seq_slots, n_new,
                                   static_cast<const __half*>(k), static_cast<const __half*>(v),
                                   as_stream(stream)));
}

int ekv_decode_attn(ekv_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_slots,
                    const void* q, void* o, void* stream) {
  if (!c || layer < 0 || layer >= c->st.L || n_seqs < 0 || n_seqs > c->st.S) return EKV_EINVAL;
  if (n_seqs == 0) return EKV_OK;
  if (!seq_slots || !q || !o) return EKV_EINVAL;
  if (((uintptr_t)q | (uintptr_t)o) & 15) return EKV_EINVAL;
  const int splits = attn_splits(c, n_seqs, c->vbits[layer]);
  if (n_seqs * c->st.Hkv * splits > c->st.attn_parts_cap) return EKV_ESTATE;
  return cuda_status(launch_decode_attn(c->st, layer, n_seqs, seq_slots,
                                        static_cast<const __half*>(q), static_cast<__half*>(o),
                                        splits, c->vbits[layer], attn_pack(c, n_seqs, c->vbits[layer]),
                                        as_stream(stream)));
}

int ekv_append_decode_attn(ekv_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_slots,
                           const void* k, const void* v, const void* q, void* o, int32_t flags,
                           void* stream) {
  if (flags & ~(EKV_AFTER_OTHER_LAYER | EKV_AFTER_PRODUCER)) return EKV_EINVAL;
  if (!c || layer < 0 || layer >= c->st.L || n_seqs < 0 || n_seqs > c->st.S) return EKV_EINVAL;
  if (n_seqs == 0) return EKV_OK;
  if (!seq_slots || !k || !v || !q || !o) return EKV_EINVAL;
  if (((uintptr_t)k | (uintptr_t)v | (uintptr_t)q | (uintptr_t)o) & 15) return EKV_EINVAL;
  const int splits = attn_splits(c, n_seqs, c->vbits[layer]);
  if (n_seqs * c->st.Hkv * splits > c->st.attn_parts_cap) return EKV_ESTATE;
  return cuda_status(launch_decode_attn(c->st, layer, n_seqs, seq_slots,
                                        static_cast<const __half*>(q), static_cast<__half*>(o),
                                        splits, c->vbits[layer], attn_pack(c, n_seqs, c->vbits[layer]),
                                        as_stream(stream), static_cast<const __half*>(k),
                                        static_cast<const __half*>(v),
                                        (flags & EKV_AFTER_PRODUCER) ? OVERLAP_DEPENDENT
                                        : (flags & EKV_AFTER_OTHER_LAYER) ? OVERLAP_INDEPENDENT
                                                                          : OVERLAP_NONE));
}

int ekv_canary_kl(ekv_cache* c, int32_t layer, int32_t n_seqs, const int32_t* seq_slots,
                  const void* q, float* delta_out, void* stream) {
  if (!c || layer < 0 || layer >= c->st.L || n_seqs <= 0 || n_seqs > c->st.S) return EKV_EINVAL;
  if (!seq_slots || !q) return EKV_EINVAL;
  return cuda_status(launch_canary(c->st, layer, 1, n_seqs, seq_slots,
                                   static_cast<const __half*>(q), 0, delta_out,
                                   as_stream(stream)));
}

int ekv_canary_kl_layers(ekv_cache* c, int32_t first_layer, int32_t n_layers, int32_t n_seqs,
                         const int32_t* seq_slots, const void* q, int64_t q_layer_stride,
                         float* delta_out, void* stream) {
  if (!c || first_layer < 0 || n_layers <= 0 || first_layer + n_layers > c->st.L ||
      n_seqs <= 0 || n_seqs > c->st.S || !seq_slots || !q || q_layer_stride < 0 ||
      n_layers > 65535)
    return EKV_EINVAL;
  if (n_layers > 1 && q_layer_stride < (int64_t)n_seqs * c->st.Hq * c->st.D) return EKV_EINVAL;
  return cuda_status(launch_canary(c->st, first_layer, n_layers, n_seqs, seq_slots,
                                   static_cast<const __half*>(q), (size_t)q_layer_stride,
                                   delta_out, as_stream(stream)));
}

int ekv_tier_update(ekv_cache* c, const float* delta, const uint8_t* layer_mask, int32_t freeze,
                    void* stream) {
  if (!c) return EKV_EINVAL;
  return cuda_status(launch_tier_update(c->st, delta, layer_mask, freeze, as_stream(stream)));
}

int ekv_set_tiers(ekv_cache* c, const uint8_t* tiers, void* stream) {
  if (!c || !tiers) return EKV_EINVAL;
  std::vector<int32_t> t(c->st.L);
  for (int l = 0; l < c->st.L; ++l) {
    if (!valid_bits(tiers[l])) return EKV_EINVAL;
    t[l] = tiers[l];
  }
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(c->st.tier, t.data(), t.size() * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // t is a host temporary
  return cuda_status(e);
}

int ekv_set_clip(ekv_cache* c, int32_t layer, const float* k_clip, const float* v_clip,
                 void* stream) {
  if (!c || layer < 0 || layer >= c->st.L) return EKV_EINVAL;
  if (c->st.asym) return EKV_EUNSUPPORTED;  // thresholds cap the symmetric quantizer's absmax
  const int H = c->st.Hkv, D = c->st.D;
  std::vector<float> kc((size_t)H * D, INFINITY), vc(H, INFINITY);
  auto take = [](const float* src, std::vector<float>& dst) {
    if (!src) return true;
    for (size_t i = 0; i < dst.size(); ++i) {
      if (!(src[i] > 0.f)) return false;  // NaN, zero and negative thresholds
      dst[i] = src[i];
    }
    return true;
  };
  if (!take(k_clip, kc) || !take(v_clip, vc)) return EKV_EINVAL;
  cudaStream_t s = as_stream(stream);
  const size_t lh = (size_t)layer * H;
  cudaError_t e = cudaMemcpyAsync(c->st.kclip + lh * D, kc.data(), kc.size() * 4,
                                  cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(c->st.vclip + lh, vc.data(), vc.size() * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);  // kc, vc are host temporaries
  return cuda_status(e);
}

int ekv_get_clip(ekv_cache* c, int32_t layer, float* k_clip, float* v_clip, void* stream) {
  if (!c || layer < 0 || layer >= c->st.L) return EKV_EINVAL;
  const int H = c->st.Hkv, D = c->st.D;
  cudaStream_t s = as_stream(stream);
  const size_t lh = (size_t)layer * H;
  cudaError_t e = cudaSuccess;
  if (k_clip)
    e = cudaMemcpyAsync(k_clip, c->st.kclip + lh * D, (size_t)H * D * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && v_clip)
    e = cudaMemcpyAsync(v_clip, c->st.vclip + lh, (size_t)H * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

int ekv_get_state(ekv_cache* c, uint8_t* tiers, float* ema, float* delta, int32_t* ema_valid,
                  void* stream) {
  if (!c) return EKV_EINVAL;
  const int L = c->st.L;
  cudaStream_t s = as_stream(stream);
  std::vector<int32_t> t(L);
  cudaError_t e = cudaMemcpyAsync(t.data(), c->st.tier, L * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && ema)
    e = cudaMemcpyAsync(ema, c->st.ema, L * 12, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && delta)
    e = cudaMemcpyAsync(delta, c->st.delta, L * 12, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && ema_valid)
    e = cudaMemcpyAsync(ema_valid, c->st.ema_valid, L * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return EKV_ECUDA;
  if (tiers)
    for (int l = 0; l < L; ++l) tiers[l] = (uint8_t)t[l];
  return EKV_OK;
}

int ekv_seq_len(ekv_cache* c, int32_t layer, int32_t seq_slot, int32_t* out, void* stream) {
  if (!c || !out || layer < 0 || layer >= c->st.L || seq_slot < 0 || seq_slot >= c->st.S)
    return EKV_EINVAL;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(out, c->st.len + ls_index(c->st, layer, seq_slot), 4,
                                  cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

int ekv_block_table(ekv_cache* c, int32_t layer, int32_t seq_slot, int32_t kv_head, int32_t* out,
                    int32_t cap, int32_t* n_out, void* stream) {
  if (!c || !n_out || layer < 0 || layer >= c->st.L || seq_slot < 0 || seq_slot >= c->st.S ||
      kv_head < 0 || kv_head >= c->st.Hkv || cap < 0 || (cap > 0 && !out))
    return EKV_EINVAL;
  int32_t len = 0;
  int rc = ekv_seq_len(c, layer, seq_slot, &len, stream);
  if (rc) return rc;
  const int nb = (len + BLOCK - 1) / BLOCK;
  *n_out = nb;
  const int n = nb < cap ? nb : cap;
  if (n == 0) return EKV_OK;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(out, c->st.bt + lsh_index(c->st, layer, seq_slot, kv_head) * c->st.maxblk,
                                  (size_t)n * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

int ekv_read_pages(ekv_cache* c, int32_t layer, int32_t seq_slot, int32_t kv_head,
                   int32_t first_block, int32_t n_blocks, void* dst, size_t dst_stride,
                   void* stream) {
  if (!c || !dst || layer < 0 || layer >= c->st.L || seq_slot < 0 || seq_slot >= c->st.S ||
      kv_head < 0 || kv_head >= c->st.Hkv || first_block < 0 || n_blocks < 0 ||
      first_block + n_blocks > c->st.maxblk || (dst_stride & 15) || ((uintptr_t)dst & 15))
    return EKV_EINVAL;
  const int vb = c->vbits[layer];
  if ((int64_t)dst_stride < page_bytes(16, vb, c->st.D, c->st.asym)) return EKV_EINVAL;
  if (n_blocks == 0) return EKV_OK;
  return cuda_status(launch_read_pages(c->st, layer, seq_slot, kv_head, first_block, n_blocks,
                                       static_cast<uint8_t*>(dst), dst_stride, as_stream(stream)));
}

int ekv_stats(ekv_cache* c, int32_t first_layer, int32_t n_layers, ekv_stats_t* out,
              void* stream) {
  if (!c || !out || first_layer < 0 || n_layers <= 0 || first_layer + n_layers > c->st.L)
    return EKV_EINVAL;
  cudaStream_t s = as_stream(stream);
  unsigned long long cnt[3 * NFMT + 1];
  std::vector<int32_t> len((size_t)n_layers * c->st.S);
  cudaError_t e = launch_stats(c->st, first_layer, n_layers, c->census, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(cnt, c->census, sizeof(cnt), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(len.data(), c->st.len + ls_index(c->st, first_layer, 0),
                        len.size() * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return EKV_ECUDA;
  if (cnt[3 * NFMT] != 0) return EKV_ESTATE;  // blocks in use without a page
  memset(out, 0, sizeof(*out));
  const int D = c->st.D;
  double kbits = 0, vbits = 0, bytes = 0;
  int64_t tokens = 0;
  for (int32_t t : len) tokens += (int64_t)t * c->st.Hkv;
  for (int f = 0; f < NFMT; ++f) {
    out->sealed_pages[f] = (int64_t)cnt[f];
    out->open_pages[f] = (int64_t)cnt[NFMT + f];
    out->open_rows[f] = (int64_t)cnt[2 * NFMT + f];
    const int kb = bits_of_code(f >> 2), vb = bits_of_code(f & 3);
    const double sealed_tok = (double)BLOCK * out->sealed_pages[f];
    kbits += sealed_tok * kb + (double)out->open_rows[f] * 16;
    vbits += (sealed_tok + (double)out->open_rows[f]) * vb;
    bytes += (double)(out->sealed_pages[f] + out->open_pages[f]) * page_bytes(kb, vb, D, c->st.asym);
  }
  out->tokens = tokens;
  if (tokens > 0) {
    out->k_bits = kbits / (double)tokens;
    out->v_bits = vbits / (double)tokens;
    out->cost_vs_c0 = (out->k_bits + out->v_bits) / 32.0;
    out->page_bytes = bytes;
    out->fp16_bytes = (double)tokens * D * 4.0;
    out->saved_vs_fp16 = 1.0 - bytes / out->fp16_bytes;
  }
  return EKV_OK;
}

int ekv_pool_free(ekv_cache* c, int32_t format, int64_t* out, void* stream) {
  if (!c || !out || format < 0 || format >= NFMT) return EKV_EINVAL;
  int32_t t = 0;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(&t, c->st.top + format, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *out = t;
  return cuda_status(e);
}

int ekv_debug_set(ekv_cache* c, int32_t knob, int64_t value) {
  if (!c) return EKV_EINVAL;
  switch (knob) {
    case EKV_DEBUG_WAIT_EXPIRY: c->st.dbg_wait_expiry = value != 0; return EKV_OK;
    default: return EKV_EINVAL;
  }
}

int ekv_sync(ekv_cache* c, void* stream) {
  if (!c) return EKV_EINVAL;
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return EKV_ECUDA;
  int32_t err = 0;
  e = cudaMemcpyAsync(&err, c->st.err, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->st.err, 0, 4, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return EKV_ECUDA;
  return err;
}

int64_t ekv_state_size(ekv_cache* c) {
  if (!c) return -1;
  return 8 + (int64_t)c->st.L * (4 + 12 + 4 + 12 + 4 + 4);
}

int ekv_state_save(ekv_cache* c, void* blob, int64_t bytes, void* stream) {
  if (!c || !blob || bytes < ekv_state_size(c)) return EKV_EINVAL;
  const int L = c->st.L;
  uint8_t* p = static_cast<uint8_t*>(blob);
  const uint32_t magic = 0x454B5632u, nl = (uint32_t)L;
  memcpy(p, &magic, 4);
  memcpy(p + 4, &nl, 4);
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(p + 8, c->st.tier, L * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p + 8 + L * 4, c->st.ema, L * 12, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p + 8 + L * 16, c->st.ema_valid, L * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p + 8 + L * 20, c->st.delta, L * 12, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p + 8 + L * 32, c->st.cand, L * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(p + 8 + L * 36, c->st.cnt, L * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

int ekv_state_load(ekv_cache* c, const void* blob, int64_t bytes, void* stream) {
  if (!c || !blob || bytes < ekv_state_size(c)) return EKV_EINVAL;
  const int L = c->st.L;
  const uint8_t* p = static_cast<const uint8_t*>(blob);
  uint32_t magic = 0, nl = 0;
  memcpy(&magic, p, 4);
  memcpy(&nl, p + 4, 4);
  if (magic != 0x454B5632u || nl != (uint32_t)L) return EKV_EINVAL;
  for (int l = 0; l < L; ++l) {
    int32_t t;
    memcpy(&t, p + 8 + 4 * l, 4);
    if (!valid_bits(t)) return EKV_EINVAL;
  }
  cudaStream_t s = as_stream(stream);
  cudaError_t e = cudaMemcpyAsync(c->st.tier, p + 8, L * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->st.ema, p + 8 + L * 4, L * 12, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->st.ema_valid, p + 8 + L * 16, L * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->st.delta, p + 8 + L * 20, L * 12, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->st.cand, p + 8 + L * 32, L * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->st.cnt, p + 8 + L * 36, L * 4, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

}  // extern "C"
