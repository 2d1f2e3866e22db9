// Host-side driver for the launch-shape decisions (csrc/launch_choice.h):
// reads lines
//   M N K in_elem_bytes layout pair multicast visible_devices forced_tile_n
//   batch dynamic_mode capped stream_k resident_units_1 resident_units_2 resident_units_4
// (pair 0: the automatic choice, made as the library makes it) and prints
// "unit tile_n tiles dynamic units waves" for each, so the CPU
// tests can check the choices the library makes for the benchmark shapes
// and the rules behind them.
#include <cstdio>

#include "launch_choice.h"

int main() {
    long long M, N, K, batch;
    int ib, layout, pair, mc, visible, forced, mode, capped, sk, r1, r2, r4;
    while (std::scanf("%lld %lld %lld %d %d %d %d %d %d %lld %d %d %d %d %d %d", &M, &N, &K, &ib, &layout, &pair,
                      &mc, &visible, &forced, &batch, &mode, &capped, &sk, &r1, &r2, &r4) == 16) {
        if (pair == 0) pair = mc == 1 ? 2 : gb300::launch_auto_pair(M, N, batch, r2, r1);
        const int unit = gb300::launch_unit_ctas(pair, mc, visible, K, ib, layout);
        const int resident = unit == 1 ? r1 : unit == 2 ? r2 : r4;
        const int bn = gb300::launch_tile_n(forced, M, N, unit, layout, batch, resident);
        long long tiles = 0;
        int units = 0, waves = 0, dyn = 0;
        if (bn > 0) {
            const long long tile_m = 128LL * unit;
            tiles = batch * ((M + tile_m - 1) / tile_m) * ((N + bn - 1) / bn);
            dyn = gb300::launch_dynamic_lists(mode, capped != 0, sk != 0, tiles, resident, &units, &waves) ? 1 : 0;
        }
        std::printf("%d %d %lld %d %d %d\n", unit, bn, tiles, dyn, units, waves);
    }
    return 0;
}
