// prefill.cu - batched prefill of a prompt chunk.
#include "qw_prefill.h"

namespace qw {

size_t prefill_workspace_bytes(const qw_config &, int) { return 256; }

cudaError_t prefill_prepare() { return cudaSuccess; }

void prefill_init(PrefillState *st, const DecodeArgs &, uint8_t *buf, size_t bytes, int rows_max, int nsm) {
    st->buf = buf;
    st->bytes = bytes;
    st->rows_max = rows_max;
    st->nsm = nsm;
    st->ready = 0;
}

int prefill_run(PrefillState *, const DecodeArgs &, int, const int32_t *, int, cudaStream_t) { return 1; }

}  // namespace qw
