// pkv_attention_d64.cu -- paged attention and combine kernels for head_dim 64.
#include "pkv_attention.cuh"

namespace pkv {
int dispatch_attention_d64(int GD, bool wide, const TMaps& tm, const AttnParams& p, long long mi, cudaStream_t st) {
    return dispatch_g<64>(GD, wide, tm, p, mi, st);
}
int combine_d64(const CombineParams& c, cudaStream_t st) { return launch_combine<64>(c, st); }
}  // namespace pkv
