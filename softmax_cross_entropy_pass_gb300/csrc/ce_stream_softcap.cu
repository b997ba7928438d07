// ce_stream_softcap.cu -- the streaming kernel's instantiations with softcap
// (and z-loss / token accuracy), aligned and ragged rows, compiled apart so
// they build in parallel with the others.
#include "ce_stream.cuh"

namespace ce {

const void *stream_kernel_softcap(int dtype, int mode, int shape, int cl, bool ragged) {
    return ragged ? stream_kernel_options_for<true, 2>(dtype, mode, shape, cl)
                  : stream_kernel_options_for<false, 2>(dtype, mode, shape, cl);
}

}  // namespace ce
