// decode_mma.cu -- the 4-bit instantiations of the register-MMA decode
// kernel (decode_mma.cuh) and the entry points, which send 8-bit weights to
// the instantiations in decode_mma8.cu.
#include "decode_mma.cuh"

namespace tmw4 {

extern template cudaError_t dm_launch_wb<8>(const GemmArgs &, const CUtensorMap &, bool, int, int, int,
                                            cudaStream_t);
extern template int dm_ctas_per_sm_wb<8>(bool, int, int, int);
extern template int dm_cluster_split_wb<8>(bool, int, int, int, int, int, int *);

template cudaError_t dm_launch_wb<4>(const GemmArgs &, const CUtensorMap &, bool, int, int, int, cudaStream_t);
template int dm_ctas_per_sm_wb<4>(bool, int, int, int);
template int dm_cluster_split_wb<4>(bool, int, int, int, int, int, int *);

int decode_mma_nt8(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : 0; }

int decode_mma_ctas_per_sm(bool bf16, int M, int group, int kgroups, int wbits) {
  return wbits == 8 ? dm_ctas_per_sm_wb<8>(bf16, M, group, kgroups) : dm_ctas_per_sm_wb<4>(bf16, M, group, kgroups);
}

int decode_mma_cluster_split(bool bf16, int M, int K, int group, int kgroups, int requested, int *kb_per_split,
                             int wbits) {
  return wbits == 8 ? dm_cluster_split_wb<8>(bf16, M, K, group, kgroups, requested, kb_per_split)
                    : dm_cluster_split_wb<4>(bf16, M, K, group, kgroups, requested, kb_per_split);
}

cudaError_t launch_decode_mma(const GemmArgs &a, const CUtensorMap &tmap_a, bool bf16, int kgroups, int grid,
                              int cluster, cudaStream_t st) {
  return a.wbits == 8 ? dm_launch_wb<8>(a, tmap_a, bf16, kgroups, grid, cluster, st)
                      : dm_launch_wb<4>(a, tmap_a, bf16, kgroups, grid, cluster, st);
}

void decode_mma_plan(int M, int N, int K, int group, int max_ctas, int *grid, long long *tiles,
                     int *slots) {
  const long long GR = K / group;
  const long long T = N / TILE_N;
  const long long U = T * GR;
  const long long G = std::max<long long>(1, std::min<long long>(max_ctas, U));
  int maxc = 1;
  for (long long t = 0; t < T; ++t) {
    const int c = cta_of_unit((t + 1) * GR - 1, U, G) - cta_of_unit(t * GR, U, G) + 1;
    if (c > maxc) maxc = c;
  }
  *grid = static_cast<int>(G);
  *tiles = T;
  *slots = maxc;
  (void)M;
}

}  // namespace tmw4
