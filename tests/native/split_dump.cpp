// Host-side driver for the split-K choice (csrc/launch_choice.h): reads lines
//   forced tiles units k_blocks slice_floats workspace_floats
// and prints the number of K slices the library would use for each.
#include <cstdio>

#include "launch_choice.h"

int main() {
    int forced;
    long long tiles, units, kb, slice, ws;
    while (std::scanf("%d %lld %lld %lld %lld %lld", &forced, &tiles, &units, &kb, &slice, &ws) == 6)
        std::printf("%d\n", gb300::launch_split_k(forced, tiles, units, kb, slice, ws));
    return 0;
}
