// prefill_tc_hd64.cu -- instantiations of the tensor-core prefill for
// head_dim 64 (G = 1..8 query heads per kv head).  One translation unit per
// head dim so the builds run in parallel.
#include "prefill_tc.cuh"

namespace slotkv {

int launch_prefill_tc_hd64(int G, const PrefillParams& p, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, unsigned ctas, cudaStream_t stream) {
    return launch_prefill_hd<64>(G, p, tmK, tmV, ctas, stream);
}

}  // namespace slotkv
