// k x k affine scans (placeholder until the kernels land).
#include "common.cuh"

namespace mg {

size_t affine_ws_bytes(int64_t, int64_t, int64_t, int, int) { return kControlBytes; }

mg_status launch_affine_fwd(const float *, const float *, float *, float *, int64_t, int64_t,
                            int64_t, int, int, void *, size_t, cudaStream_t, const LaunchOpts &)
{
    return fail(MG_ERR_UNSUPPORTED, "mg_affine_scan_fwd: not built yet");
}

mg_status launch_affine_bwd(const float *, const float *, const float *, const float *,
                            const float *, float *, float *, int64_t, int64_t, int64_t, int, int,
                            void *, size_t, cudaStream_t, const LaunchOpts &)
{
    return fail(MG_ERR_UNSUPPORTED, "mg_affine_scan_bwd: not built yet");
}

}  // namespace mg
