// Backward instantiations of the staged kernels (sms_tile.cuh).
#include "sms_tile.cuh"

namespace sms {

bool cta_fits_bwd(int64_t cols, int dtype, bool aligned)
{
    return tile::row_vectors(cols, dtype, aligned) <= tile::tile_capacity(dtype, true);
}

cudaError_t launch_bwd_cta(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    FwdArgs none = {};
    return tile::dispatch<true>(none, a, a.cols, dtype, aligned, st);
}

}  // namespace sms
