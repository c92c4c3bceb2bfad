// Instantiations of the SIMT kernel, part a of 5 (split only to compile in
// parallel).
#include "simt_kernel.cuh"

namespace gemm_f32 {
namespace simt_detail {

extern const SimtEntry kSimtPartA[] = {
    {{128, 128, 16, 8, 8, 2, false}, launch_cfg<128, 128, 16, 8, 8, 2>},
    {{64, 64, 16, 4, 4, 2, false}, launch_cfg<64, 64, 16, 4, 4, 2>},
    {{64, 64, 32, 4, 4, 2, false}, launch_cfg<64, 64, 32, 4, 4, 2>},
    {{128, 64, 16, 8, 4, 2, false}, launch_cfg<128, 64, 16, 8, 4, 2>},
    {{32, 32, 64, 4, 4, 2, false}, launch_cfg<32, 32, 64, 4, 4, 2>},
    // barrier-coalescing ablation: A and B published separately
    {{128, 128, 16, 8, 8, 2, true}, launch_cfg<128, 128, 16, 8, 8, 2, true>},
    {{64, 64, 16, 4, 4, 1, true}, launch_cfg<64, 64, 16, 4, 4, 1, true>},
};
extern const int kSimtPartACount = (int)(sizeof(kSimtPartA) / sizeof(kSimtPartA[0]));

}  // namespace simt_detail
}  // namespace gemm_f32
