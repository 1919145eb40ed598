// decode_g1.cu - decode kernel instantiations with the SMs as one group.
#include "decode_kernel.cuh"

namespace qw {

const void *decode_fn_d1(int fmt, int kv_f32) {
    if (fmt == 1) return kv_f32 ? (const void *)decode_kernel<1, true, float> : (const void *)decode_kernel<1, true, __nv_bfloat16>;
    return kv_f32 ? (const void *)decode_kernel<1, false, float> : (const void *)decode_kernel<1, false, __nv_bfloat16>;
}

size_t decode_smem_bytes_impl() { return sizeof(Smem); }

}  // namespace qw
