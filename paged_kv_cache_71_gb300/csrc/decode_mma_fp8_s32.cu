// decode_mma_fp8_s32.cu -- tensor-core decode instantiations for an FP8 E4M3 K/V cache (128-dim heads, bf16 queries),
// block size 32.  (One file per cache dtype and block size, so that the instantiations compile in parallel.)
#include "decode_mma.cuh"

namespace pkv {

#define PKV_INST(G_, HP_)                                                                                   \
    template cudaError_t launch_paged_decode_mma<G_, 32, KvE4M3, HP_>(const CUtensorMap&, const CUtensorMap&,     \
                                                                  const DecodeArgs&, int, int, size_t, cudaStream_t);
PKV_INST(1, 1)
PKV_INST(2, 1)
PKV_INST(4, 1)
PKV_INST(8, 1)
PKV_INST(1, 2)
PKV_INST(2, 2)
PKV_INST(4, 2)
PKV_INST(8, 2)
#undef PKV_INST

}  // namespace pkv
