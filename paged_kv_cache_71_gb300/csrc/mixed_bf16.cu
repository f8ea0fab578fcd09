// mixed_bf16.cu -- mixed-step kernel instantiations (mixed.cuh) for a bf16 K/V cache, 16-token blocks, GQA groups
// 1, 2, 4 and 8.  (One file per cache dtype, so that the instantiations compile in parallel.)
#include "mixed.cuh"

namespace pkv {

#define PKV_INST(G_)                                                                                        \
    template cudaError_t launch_paged_mixed<0, G_, KvBF16>(const CUtensorMap&, const CUtensorMap&,             \
                                                         const CUtensorMap&, const PrefillArgs&,               \
                                                         const DecodeArgs&, const MixedArgs&, int, size_t,     \
                                                         cudaStream_t);
PKV_INST(1)
PKV_INST(2)
PKV_INST(4)
PKV_INST(8)
#undef PKV_INST

}  // namespace pkv
