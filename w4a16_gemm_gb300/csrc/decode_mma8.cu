// decode_mma8.cu -- the 8-bit (int8 with a zero point, FP8 E4M3)
// instantiations of the register-MMA decode kernel (decode_mma.cuh).
#include "decode_mma.cuh"

namespace tmw4 {

template cudaError_t dm_launch_wb<8>(const GemmArgs &, const CUtensorMap &, bool, int, int, int, cudaStream_t);
template int dm_ctas_per_sm_wb<8>(bool, int, int, int);
template int dm_cluster_split_wb<8>(bool, int, int, int, int, int, int *);

}  // namespace tmw4
