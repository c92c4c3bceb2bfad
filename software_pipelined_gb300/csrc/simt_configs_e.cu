// Instantiations of the SIMT kernel, part e of 5: fragments handed out by warp
// shuffles instead of broadcast shared-memory loads (the fragment-load
// ablation), on the tiles the dispatcher uses.
#include "simt_kernel.cuh"

namespace gemm_f32 {
namespace simt_detail {

extern const SimtEntry kSimtPartE[] = {
    {{128, 128, 16, 8, 8, 2, false, 1, true}, launch_cfg<128, 128, 16, 8, 8, 2, false, 1, true>},
    {{64, 64, 16, 4, 4, 2, false, 1, true}, launch_cfg<64, 64, 16, 4, 4, 2, false, 1, true>},
    {{64, 64, 16, 4, 4, 4, false, 2, true}, launch_cfg<64, 64, 16, 4, 4, 4, false, 2, true>},
    {{32, 32, 32, 4, 4, 3, false, 4, true}, launch_cfg<32, 32, 32, 4, 4, 3, false, 4, true>},
    {{32, 32, 64, 4, 4, 3, false, 4, true}, launch_cfg<32, 32, 64, 4, 4, 3, false, 4, true>},
};
extern const int kSimtPartECount = (int)(sizeof(kSimtPartE) / sizeof(kSimtPartE[0]));

}  // namespace simt_detail
}  // namespace gemm_f32
