// codec_tc.cu -- tensor-core (tcgen05) encode/decode for bf16, d = 128.
#include "spectra_internal.cuh"

namespace spectra {

spectra_status launch_tc_images(const spectra_plan*, cudaStream_t) { return SPECTRA_OK; }

spectra_status launch_encode_tc(const spectra_plan*, const void*, int, int64_t, int64_t, uint8_t*,
                                int64_t, float*, int64_t, cudaStream_t, bool* done)
{
    *done = false;
    return SPECTRA_OK;
}

spectra_status launch_decode_tc(const spectra_plan*, const uint8_t*, int64_t, const float*, int64_t,
                                int64_t, void*, int, int64_t, cudaStream_t, bool* done)
{
    *done = false;
    return SPECTRA_OK;
}

}  // namespace spectra
