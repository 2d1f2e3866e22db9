// Host-side driver for the kernel's work schedule (csrc/schedule.h): reads
// "tiles units kblocks allow_stream_k" lines on stdin and prints, for each,
// the schedule and every unit's work items, so the CPU tests can check that
// every (tile, k-block) is covered exactly once and the stream-K bookkeeping
// (contributor roles, slots, flags) is consistent.  A line "tiles units
// waves -1" prints the lists of a dynamic work list instead.
#include <cstdio>

#include "schedule.h"

int main() {
    int tiles, units, kb, allow;
    while (std::scanf("%d %d %d %d", &tiles, &units, &kb, &allow) == 4) {
        if (allow < 0) {   // a dynamic work list: tiles, units, waves (= kb), -1
            const int n = gb300::dyn_list_count(tiles, units, kb);
            std::printf("D %d %d %d %d\n", tiles, units, kb, n);
            for (int c = 0; c < n; ++c)
                for (int k = 0; k < gb300::dyn_list_len(c, units, kb); ++k)
                    std::printf("L %d %d %d\n", c, k, gb300::dyn_list_tile(c, k, units, kb));
            std::printf("E\n");
            continue;
        }
        const gb300::Schedule s = gb300::make_schedule(tiles, units, kb, allow != 0);
        std::printf("S %d %d %d %d %d\n", s.tiles, s.units, s.kb, s.dp_waves, s.sk_tiles);
        for (int u = 0; u < s.units; ++u) {
            const int n = gb300::work_count(s, u);
            for (int j = 0; j < n; ++j) {
                const gb300::Work w = gb300::work_item(s, u, j);
                std::printf("W %d %d %d %d %d %d %d %d %d\n", u, j, w.tile, w.kb_begin, w.kb_end, w.contrib,
                            w.ncontrib, w.slot, w.sk_index);
            }
        }
        std::printf("E\n");
    }
    return 0;
}
