// Chunked-prefill causal attention (tcgen05 / TMEM).  Placeholder until the
// tensor-core kernel lands: reports UNSUPPORTED.
#include "kvattn_internal.cuh"

namespace kvattn {

kvattn_status launch_prefill(const PrefillArgs& a, cudaStream_t s)
{
    (void)a;
    (void)s;
    return KVATTN_ERR_UNSUPPORTED;
}

}  // namespace kvattn
