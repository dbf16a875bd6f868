// Forward instantiations of the staged kernels (sms_tile.cuh).
#include "sms_tile.cuh"

namespace sms {

bool cta_fits(int64_t cols, int dtype, bool aligned)
{
    return tile::row_vectors(cols, dtype, aligned) <= tile::tile_capacity(dtype, false);
}

cudaError_t launch_fwd_cta(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    BwdArgs none = {};
    return tile::dispatch<false>(a, none, a.cols, dtype, aligned, st);
}

}  // namespace sms
