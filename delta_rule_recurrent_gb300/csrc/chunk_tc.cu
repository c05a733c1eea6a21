// chunk_tc.cu -- chunkwise delta-rule forward on tcgen05 tensor cores.
#include "dn_common.cuh"
#include "dn_internal.h"

namespace dn {

bool chunk_tc_supports(int dk, int dv, int dt) {
    (void)dk; (void)dv; (void)dt;
    return false;
}

cudaError_t launch_chunk_tc(const void*, const void*, const void*, const void*, const float*,
                            void*, float*, int, int, int, int, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace dn
