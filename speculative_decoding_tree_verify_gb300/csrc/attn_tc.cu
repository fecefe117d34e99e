// attn_tc.cu -- tensor-core (tcgen05) tree-masked attention.  Shapes it does not take go to the
// CUDA-core kernel (attn_simt.cu).
#include "sv_internal.cuh"

namespace sv {

size_t attn_workspace_size(int B, int T, int Hq, int Hkv, int D, int kv_cap) {
    (void)B; (void)T; (void)Hq; (void)Hkv; (void)D; (void)kv_cap;
    return 0;
}

bool attn_tc_supported(const AttnArgs& a) {
    (void)a;
    return false;
}

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s) {
    (void)a; (void)s;
    return cudaErrorNotSupported;
}

}  // namespace sv
