// decode_i8_s4.cu -- paged decode kernel instantiations for a symmetric INT8 K/V cache (per-tensor scale) with bf16 queries,
// block size 4.  (One file per cache dtype and block size, so that the
// instantiations compile in parallel.)
#include "decode.cuh"

namespace pkv {

#define PKV_INST(G_, D_)                                                                                     \
    template cudaError_t launch_paged_decode<G_, D_, 4, KvI8, KvBF16>(                                       \
        const CUtensorMap&, const CUtensorMap&, const DecodeArgs&, int, int, size_t, cudaStream_t);
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
