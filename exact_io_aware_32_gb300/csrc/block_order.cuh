// Order in which the CTAs of one attention kernel visit (head, block) pairs.
#pragma once

namespace fa {

// CTAs start roughly in increasing linear index. With the head as the fastest
// coordinate, the CTAs resident at one time would belong to as many heads as
// there are SMs, and the tiles they stream (K/V, or Q/dO) would leave L2
// before the other CTAs of the same head come to read them. So the heads go in
// groups of 'group' (about one wave of CTAs): inside a group the block index
// is the slow coordinate, so the heaviest blocks of the group start first, and
// all CTAs of a head run at about the same time and share its tiles in L2.
// (head, block) of the linear index in that order.
__device__ __forceinline__ void grouped_index(int linear, int BH, int nblk, int group, int& bh, int& blk) {
  const int per_group = group * nblk;
  const int g = linear / per_group;
  const int idx = linear - g * per_group;
  const int gsize = min(group, BH - g * group);  // the last group may be smaller
  blk = idx / gsize;
  bh = g * group + (idx - blk * gsize);
}

}  // namespace fa
