// ekv_attn_asym.cu — decode attention over pages of the KIVI-style asymmetric
// quantizer: the kernels of ekv_attn_body.cuh instantiated with EKV_ATTN_ASYM 1
// (a translation unit of its own, so both variants compile in parallel).
#define EKV_ATTN_ASYM 1
#include "ekv_attn_body.cuh"
