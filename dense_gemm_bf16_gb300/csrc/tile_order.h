// Tile order of the GEMM kernels (host and device).
//
// Output tiles are visited in groups of `group_m` tile-rows: inside a group
// the walk goes down the group's tile-rows first and then to the next
// tile-column, so the CTAs running at the same time share B tiles (and A
// tiles across consecutive columns) in L2.  This is the grouped ordering of
// "Skill: Write a Triton GEMM Kernel", Required reasoning process step 2, and
// of "GEMM Kernel Optimization", L2 Cache Grouping; group_m = 1 gives the
// plain row-major tile order.  The map t -> (pid_m, pid_n) is a bijection on
// [0, num_pid_m * num_pid_n) for every group_m >= 1 (the last, partial group
// is walked with its own height).
#pragma once

#ifdef __CUDACC__
#define DG_HD __host__ __device__ __forceinline__
#else
#define DG_HD inline
#endif

namespace dg {

DG_HD void tile_coord(int t, int num_pid_m, int num_pid_n, int group_m, int& pid_m, int& pid_n) {
    const int in_group = group_m * num_pid_n;
    const int group_id = t / in_group;
    const int first_m = group_id * group_m;
    const int rest = num_pid_m - first_m;
    const int height = rest < group_m ? rest : group_m;
    pid_m = first_m + (t % height);
    pid_n = (t % in_group) / height;
}

}  // namespace dg
