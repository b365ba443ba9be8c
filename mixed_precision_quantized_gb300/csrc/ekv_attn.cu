// ekv_attn.cu — decode attention over pages of the symmetric quantizer (the
// kernels of ekv_attn_body.cuh instantiated with EKV_ATTN_ASYM 0), and the
// entry points that pick a handle's variant.
#define EKV_ATTN_ASYM 0
#include "ekv_attn_body.cuh"

namespace ekv {

int attn_ctas_per_sm(int) { return 1; }

namespace {
bool g_pack2_ok = true;  // two half-size CTAs fit on an SM (checked by attn_init)
}

bool attn_pack2_ok() { return g_pack2_ok; }

cudaError_t attn_init() {
  bool ok = true;
  cudaError_t e = attn_init_sym(&ok);
  if (e == cudaSuccess) e = attn_init_asym(&ok);
  g_pack2_ok = ok;
  return e;
}

cudaError_t launch_decode_attn(const DevState& st, int layer, int n_seqs, const int32_t* slots,
                               const __half* q, __half* o, int splits, int vb, int pack,
                               cudaStream_t s, const __half* knew, const __half* vnew,
                               int overlap) {
  return (st.asym ? launch_decode_attn_asym : launch_decode_attn_sym)(
      st, layer, n_seqs, slots, q, o, splits, vb, pack, s, knew, vnew, overlap);
}

}  // namespace ekv
