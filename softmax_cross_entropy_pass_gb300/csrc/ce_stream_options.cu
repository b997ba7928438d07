// ce_stream_options.cu -- the streaming kernel's instantiations with z-loss
// and token accuracy (no softcap) for aligned rows; the ragged ones are in
// ce_stream_options_ragged.cu, so the two build in parallel with the others.
#include "ce_stream.cuh"

namespace ce {

const void *stream_kernel_options(int dtype, int mode, int shape, int cl, bool ragged) {
    return ragged ? stream_kernel_options_ragged(dtype, mode, shape, cl)
                  : stream_kernel_options_for<false, 1>(dtype, mode, shape, cl);
}

}  // namespace ce
