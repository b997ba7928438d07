// ce_stream_options_ragged.cu -- the streaming kernel's instantiations with
// z-loss and token accuracy (no softcap) for rows that do not all start on a
// 16-byte boundary.
#include "ce_stream.cuh"

namespace ce {

const void *stream_kernel_options_ragged(int dtype, int mode, int shape, int cl) {
    return stream_kernel_options_for<true, 1>(dtype, mode, shape, cl);
}

}  // namespace ce
