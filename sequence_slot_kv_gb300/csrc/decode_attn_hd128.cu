// decode_attn_hd128.cu -- instantiations of the fused decode attention kernel
// for head_dim 128 (G = 1..8 query heads per kv head), and of the
// small-call kernel.  One translation unit
// per head dim so the builds run in parallel.
#include "decode_attn.cuh"
#include "decode_small.cuh"

namespace slotkv {

int launch_decode_hd128(int G, const DecodeParams& p, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, unsigned ctas, cudaStream_t stream) {
    return launch_hd<128>(G, p, tmK, tmV, ctas, stream);
}

int launch_small_hd128(int G, const DecodeParams& p, cudaStream_t stream) {
    return launch_small_hd<128>(G, p, stream);
}

}  // namespace slotkv
