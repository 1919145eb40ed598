// decode_g2.cu - decode kernel instantiations with the SMs split into two groups (one per die).
#include "decode_kernel.cuh"

namespace qw {

const void *decode_fn_d2(int fmt, int kv_f32) {
    if (fmt == 1) return kv_f32 ? (const void *)decode_kernel<2, true, float> : (const void *)decode_kernel<2, true, __nv_bfloat16>;
    return kv_f32 ? (const void *)decode_kernel<2, false, float> : (const void *)decode_kernel<2, false, __nv_bfloat16>;
}

}  // namespace qw
