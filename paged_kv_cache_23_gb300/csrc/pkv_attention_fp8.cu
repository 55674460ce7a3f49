// pkv_attention_fp8.cu -- paged attention over FP8 pools (head_dim 128): e4m3
// or e5m2 codes, a scale per kv head or per (block, kv head) tile.
#include "pkv_attention.cuh"

namespace pkv {
int dispatch_attention_fp8_d128(int fq, const TMaps& tm, const AttnParams& p, long long mi, cudaStream_t st) {
    switch (fq) {
        case 1: return launch_attention<128, 0, true, false, 1, 1>(tm, p, mi, st);
        case 2: return launch_attention<128, 0, true, false, 1, 2>(tm, p, mi, st);
        case 3: return launch_attention<128, 0, true, false, 1, 3>(tm, p, mi, st);
        default: return launch_attention<128, 0, true, false, 1, 0>(tm, p, mi, st);
    }
}
}  // namespace pkv
