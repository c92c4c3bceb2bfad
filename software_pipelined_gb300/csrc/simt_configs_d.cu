// Instantiations of the SIMT kernel, part d of 5: K split inside the CTA
// (sliced K) for the small and skinny shapes, whose grids hold too few warps.
#include "simt_kernel.cuh"

namespace gemm_f32 {
namespace simt_detail {

extern const SimtEntry kSimtPartD[] = {
    {{64, 64, 16, 4, 4, 3, false, 2}, launch_cfg<64, 64, 16, 4, 4, 3, false, 2>},
    {{64, 64, 16, 4, 4, 2, false, 2}, launch_cfg<64, 64, 16, 4, 4, 2, false, 2>},
    {{64, 64, 32, 4, 4, 2, false, 2}, launch_cfg<64, 64, 32, 4, 4, 2, false, 2>},
    {{64, 64, 32, 4, 4, 2, false, 4}, launch_cfg<64, 64, 32, 4, 4, 2, false, 4>},
    {{32, 32, 64, 4, 4, 1, false, 4}, launch_cfg<32, 32, 64, 4, 4, 1, false, 4>},
    {{32, 32, 64, 4, 4, 2, false, 4}, launch_cfg<32, 32, 64, 4, 4, 2, false, 4>},
    {{32, 32, 32, 4, 4, 2, false, 2}, launch_cfg<32, 32, 32, 4, 4, 2, false, 2>},
    {{32, 32, 32, 4, 4, 2, false, 4}, launch_cfg<32, 32, 32, 4, 4, 2, false, 4>},
    {{32, 64, 32, 4, 4, 2, false, 2}, launch_cfg<32, 64, 32, 4, 4, 2, false, 2>},
    {{64, 32, 32, 4, 4, 2, false, 2}, launch_cfg<64, 32, 32, 4, 4, 2, false, 2>},
    // deeper rings: a small tile's FFMAs per K-tile are too few to cover a copy
    {{32, 32, 32, 4, 4, 3, false, 4}, launch_cfg<32, 32, 32, 4, 4, 3, false, 4>},
    {{32, 32, 32, 4, 4, 4, false, 4}, launch_cfg<32, 32, 32, 4, 4, 4, false, 4>},
    // half-height / half-width tiles: twice the CTAs, two to an SM, for grids
    // of 32x32 tiles just over the SM count
    {{16, 32, 32, 4, 4, 3, false, 4}, launch_cfg<16, 32, 32, 4, 4, 3, false, 4>},
    {{16, 32, 32, 4, 4, 3, false, 2}, launch_cfg<16, 32, 32, 4, 4, 3, false, 2>},
    {{32, 16, 32, 4, 4, 3, false, 4}, launch_cfg<32, 16, 32, 4, 4, 3, false, 4>},
    {{32, 16, 32, 4, 4, 3, false, 2}, launch_cfg<32, 16, 32, 4, 4, 3, false, 2>},
    {{32, 32, 64, 4, 4, 3, false, 4}, launch_cfg<32, 32, 64, 4, 4, 3, false, 4>},
    {{64, 64, 16, 4, 4, 4, false, 2}, launch_cfg<64, 64, 16, 4, 4, 4, false, 2>},
    {{32, 64, 32, 4, 4, 3, false, 2}, launch_cfg<32, 64, 32, 4, 4, 3, false, 2>},
    {{64, 32, 32, 4, 4, 3, false, 2}, launch_cfg<64, 32, 32, 4, 4, 3, false, 2>},
};
extern const int kSimtPartDCount = (int)(sizeof(kSimtPartD) / sizeof(kSimtPartD[0]));

}  // namespace simt_detail
}  // namespace gemm_f32
