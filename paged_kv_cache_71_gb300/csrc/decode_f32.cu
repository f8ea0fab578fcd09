// decode_f32.cu -- instantiations of the paged decode kernel for a fp32 K/V cache, fp32 queries.
// (One file per cache dtype so that the instantiations compile in parallel.)
#include "decode.cuh"

namespace pkv {

#define PKV_INST(G_, D_)                                                                                     \
    template cudaError_t launch_paged_decode<G_, D_, KvF32, KvF32>(const CUtensorMap&, const CUtensorMap&,       \
                                                                 const DecodeArgs&, int, int, size_t,           \
                                                                 cudaStream_t);
PKV_INST(1, 64)
PKV_INST(2, 64)
PKV_INST(4, 64)
PKV_INST(8, 64)
PKV_INST(1, 128)
PKV_INST(2, 128)
PKV_INST(4, 128)
PKV_INST(8, 128)
#undef PKV_INST

}  // namespace pkv
