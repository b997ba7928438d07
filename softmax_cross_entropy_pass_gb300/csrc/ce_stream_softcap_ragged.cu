// ce_stream_softcap_ragged.cu -- the streaming kernel's instantiations with
// softcap (and z-loss / token accuracy) for rows that do not all start on a
// 16-byte boundary.
#include "ce_stream.cuh"

namespace ce {

const void *stream_kernel_softcap_ragged(int dtype, int mode, int shape, int cl) {
    return stream_kernel_options_for<true, 2>(dtype, mode, shape, cl);
}

}  // namespace ce
