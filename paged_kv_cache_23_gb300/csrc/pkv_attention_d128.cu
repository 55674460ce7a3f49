// pkv_attention_d128.cu -- paged attention (bf16 and e4m3 pools) and combine kernels for head_dim 128.
#include "pkv_attention.cuh"

namespace pkv {
int dispatch_attention_d128(int GD, bool tc, bool wide, const TMaps& tm, const AttnParams& p, long long mi,
                            cudaStream_t st) {
    if (tc) return launch_attention<128, 0, false, true, 3>(tm, p, mi, st);
    return dispatch_g<128>(GD, wide, tm, p, mi, st);
}
int combine_d128(const CombineParams& c, cudaStream_t st) { return launch_combine<128>(c, st); }

}  // namespace pkv
