// SIMT FFMA GEMM: the table of compiled configurations and its lookup.  The
// kernel is simt_kernel.cuh; its instantiations are in simt_configs_*.cu.
#include <cstdint>

#include "simt_kernel.cuh"

namespace gemm_f32 {
namespace simt_detail {
extern const SimtEntry kSimtPartA[];
extern const int kSimtPartACount;
extern const SimtEntry kSimtPartB[];
extern const int kSimtPartBCount;
extern const SimtEntry kSimtPartC[];
extern const int kSimtPartCCount;
extern const SimtEntry kSimtPartD[];
extern const int kSimtPartDCount;
extern const SimtEntry kSimtPartE[];
extern const int kSimtPartECount;
}  // namespace simt_detail

namespace {

using simt_detail::SimtEntry;

const SimtEntry& entry(int id)
{
    using namespace simt_detail;
    if (id < kSimtPartACount) return kSimtPartA[id];
    id -= kSimtPartACount;
    if (id < kSimtPartBCount) return kSimtPartB[id];
    id -= kSimtPartBCount;
    if (id < kSimtPartCCount) return kSimtPartC[id];
    id -= kSimtPartCCount;
    if (id < kSimtPartDCount) return kSimtPartD[id];
    return kSimtPartE[id - kSimtPartDCount];
}

}  // namespace

int simt_num_configs()
{
    using namespace simt_detail;
    return kSimtPartACount + kSimtPartBCount + kSimtPartCCount + kSimtPartDCount + kSimtPartECount;
}
const SimtConfig& simt_config(int id) { return entry(id).cfg; }
int simt_find_config(int bm, int bn, int stages, bool sep, int bk, int ksl, bool shfl)
{
    // bk == 0: the shallowest K-tile compiled for this tile, ring and slicing
    int best = -1;
    for (int i = 0; i < simt_num_configs(); ++i) {
        const SimtConfig& c = entry(i).cfg;
        if (c.bm != bm || c.bn != bn || c.stages != stages || c.sep != sep || c.ksl != ksl || c.shfl != shfl)
            continue;
        if (bk != 0 && c.bk != bk) continue;
        if (best < 0 || c.bk < entry(best).cfg.bk) best = i;
    }
    return best;
}

cudaError_t simt_launch(int config_id, const SimtArgs& a, cudaStream_t s)
{
    if (config_id < 0 || config_id >= simt_num_configs()) return cudaErrorInvalidValue;
    return entry(config_id).fn(a, s);
}

}  // namespace gemm_f32
