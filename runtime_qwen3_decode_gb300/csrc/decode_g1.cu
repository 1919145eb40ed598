// decode_g1.cu - decode kernel instantiations with the SMs as one group.
#include "decode_kernel.cuh"

namespace qw {

// fmt: 0 bf16 weights, 1 int8 g32 weights x f32 activations, 2 int8 g32 weights x int8 activations
const void *decode_fn_d1(int fmt, int kv_f32) {
    if (fmt == 2)
        return kv_f32 ? (const void *)decode_kernel<1, 2, float> : (const void *)decode_kernel<1, 2, __nv_bfloat16>;
    if (fmt == 1)
        return kv_f32 ? (const void *)decode_kernel<1, 1, float> : (const void *)decode_kernel<1, 1, __nv_bfloat16>;
    return kv_f32 ? (const void *)decode_kernel<1, 0, float> : (const void *)decode_kernel<1, 0, __nv_bfloat16>;
}

size_t decode_smem_bytes_impl() { return sizeof(Smem); }

}  // namespace qw
