// Instantiations of the SIMT kernel, part c of 5 (split only to compile in
// parallel).
#include "simt_kernel.cuh"

namespace gemm_f32 {
namespace simt_detail {

extern const SimtEntry kSimtPartC[] = {
    {{128, 128, 16, 8, 8, 1, false}, launch_cfg<128, 128, 16, 8, 8, 1>},
    {{64, 64, 16, 4, 4, 1, false}, launch_cfg<64, 64, 16, 4, 4, 1>},
    {{32, 32, 32, 4, 4, 1, false}, launch_cfg<32, 32, 32, 4, 4, 1>},
    {{32, 32, 64, 4, 4, 1, false}, launch_cfg<32, 32, 64, 4, 4, 1>},
    {{64, 32, 32, 4, 4, 2, false}, launch_cfg<64, 32, 32, 4, 4, 2>},
    {{64, 64, 16, 4, 4, 2, true}, launch_cfg<64, 64, 16, 4, 4, 2, true>},
    {{32, 32, 32, 4, 4, 1, true}, launch_cfg<32, 32, 32, 4, 4, 1, true>},
};
extern const int kSimtPartCCount = (int)(sizeof(kSimtPartC) / sizeof(kSimtPartC[0]));

}  // namespace simt_detail
}  // namespace gemm_f32
