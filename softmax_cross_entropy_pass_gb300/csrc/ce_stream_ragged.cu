// ce_stream_ragged.cu -- the streaming kernel's instantiations for rows
// that do not all start on a 16-byte boundary (compiled apart from the
// aligned ones so the two halves build in parallel).
#include "ce_stream.cuh"

namespace ce {

const void *stream_kernel_ragged(int dtype, int mode, int shape, int cl) {
    return stream_kernel_for<true>(dtype, mode, shape, cl);
}

}  // namespace ce
