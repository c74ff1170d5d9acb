// grid_order.cuh -- order of the CTAs of a grid over (plane, block) pairs.
//
// A plane is one (head, batch) (or key/value head, batch); its blocks are
// the query (or key) tiles a CTA owns.  With causal masking the blocks of a
// plane differ in length, and the GPU starts CTAs in index order.  Taking
// planes one at a time (each plane's longest block first) leaves the last
// plane's longest blocks to start near the end of the grid, where nothing
// else is left to overlap them.  Here planes are taken in groups: inside a
// group all planes' rank-0 blocks come first, then the rank-1 blocks, and so
// on, so a group's longest blocks start while the rest of the group's work is
// still queued; a group holds few enough planes that their K/V (or Q/dO)
// stay in L2 together.  The caller maps rank to a block (longest first).
#pragma once

namespace fa {

// Group size for `blocks` blocks per plane on `sms` SMs: about four waves
// of blocks per group, so that a group's work on all SMs lasts well beyond
// one plane's longest block (about 2 / blocks of a plane's causal work);
// measured against three waves: headline forward +2.7 %, backward +1 %,
// long-sequence backward +1 %, training-shape backward -1.5 %.  The planes are then
// spread evenly over the groups that size implies: a small last group would
// start its planes' longest blocks near the end of the grid, where nothing
// is left to overlap them (with 32 planes, groups of 15, 15 and 2 left the
// SMs idle for a sixth of a grouped-query backward; 11, 11 and 10 do not).
inline int grid_group_planes(int planes, int blocks, int sms) {
    int g = (4 * sms + blocks - 1) / (blocks > 0 ? blocks : 1);
    if (g < 1) g = 1;
    if (g > planes) g = planes;
    const int ngroups = (planes + g - 1) / g;
    return (planes + ngroups - 1) / ngroups;
}

// CTA index -> plane and rank within the plane (rank 0 starts first).
__host__ __device__ __forceinline__ void grid_decode(int idx, int planes, int blocks, int group, int &plane, int &rank) {
    const int per = group * blocks;
    const int grp = idx / per;
    const int r = idx - grp * per;
    const int rest = planes - grp * group;
    const int gp = rest < group ? rest : group;
    rank = r / gp;
    plane = grp * group + (r - rank * gp);
}

}  // namespace fa
