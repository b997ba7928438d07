// ce_stream_softcap.cu -- the streaming kernel's instantiations with softcap
// (and z-loss / token accuracy) for aligned rows; the ragged ones are in
// ce_stream_softcap_ragged.cu, so the two build in parallel with the others.
#include "ce_stream.cuh"

namespace ce {

const void *stream_kernel_softcap(int dtype, int mode, int shape, int cl, bool ragged) {
    return ragged ? stream_kernel_softcap_ragged(dtype, mode, shape, cl)
                  : stream_kernel_options_for<false, 2>(dtype, mode, shape, cl);
}

}  // namespace ce
