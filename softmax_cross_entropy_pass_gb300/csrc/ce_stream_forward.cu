// ce_stream_forward.cu -- the streaming kernel's forward-only instantiations
// (ce_forward): one CTA per row, three CTAs per SM, no class-weighted
// smoothing and no options; aligned and ragged rows.
#include "ce_stream.cuh"

namespace ce {

template <int DT, bool RAG>
static const void *forward_fn(int mode) {
    return mode == 0 ? reinterpret_cast<const void *>(&ce_stream_kernel<DT, 0, 2, 1, RAG, 3>)
                     : reinterpret_cast<const void *>(&ce_stream_kernel<DT, 1, 2, 1, RAG, 3>);
}

const void *stream_kernel_forward(int dtype, int mode, bool ragged) {
    if (mode != 0 && mode != 1) return nullptr;
    if (ragged)
        return dtype == CE_DT_F32 ? forward_fn<CE_DT_F32, true>(mode)
             : dtype == CE_DT_BF16 ? forward_fn<CE_DT_BF16, true>(mode) : forward_fn<CE_DT_F16, true>(mode);
    return dtype == CE_DT_F32 ? forward_fn<CE_DT_F32, false>(mode)
         : dtype == CE_DT_BF16 ? forward_fn<CE_DT_BF16, false>(mode) : forward_fn<CE_DT_F16, false>(mode);
}

}  // namespace ce
