// Instantiations of the SIMT kernel, part b of 5 (split only to compile in
// parallel).
#include "simt_kernel.cuh"

namespace gemm_f32 {
namespace simt_detail {

extern const SimtEntry kSimtPartB[] = {
    {{128, 128, 16, 8, 8, 3, false}, launch_cfg<128, 128, 16, 8, 8, 3>},
    {{64, 64, 16, 4, 4, 3, false}, launch_cfg<64, 64, 16, 4, 4, 3>},
    {{32, 32, 32, 4, 4, 2, false}, launch_cfg<32, 32, 32, 4, 4, 2>},
    // small, latency-bound products: more of K in flight at once
    {{32, 32, 32, 4, 4, 3, false}, launch_cfg<32, 32, 32, 4, 4, 3>},
    {{32, 64, 32, 4, 4, 2, false}, launch_cfg<32, 64, 32, 4, 4, 2>},
    {{128, 128, 16, 8, 8, 1, true}, launch_cfg<128, 128, 16, 8, 8, 1, true>},
    {{32, 32, 32, 4, 4, 2, true}, launch_cfg<32, 32, 32, 4, 4, 2, true>},
};
extern const int kSimtPartBCount = (int)(sizeof(kSimtPartB) / sizeof(kSimtPartB[0]));

}  // namespace simt_detail
}  // namespace gemm_f32
