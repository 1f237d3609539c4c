// Host-only dump of the selection's staging rule (select_stages_keys,
// select_smem_bytes in csrc/kvev_internal.h): for a launch over `launch`
// keys per sequence cut into `cl` chunks, whether its CTAs stage their keys
// in shared memory and how many bytes the launch reserves, so a CPU test can
// check that no shorter sequence of the launch stages more than that.
#include <cstdio>

#include "../decoding_kv_cache_split_gb300/csrc/kvev_internal.h"

int main() {
    const int cls[] = {1, 8};
    const int launches[] = {1, 2, 100, 8191, 10240, 10241, 20480, 81920, 81921, 81928, 90000,
                            131072, 262144};
    for (int cl : cls)
        for (int n : launches)
            std::printf("%d %d %d %zu %d\n", cl, n, kvev::select_stages_keys(n, cl) ? 1 : 0,
                        kvev::select_smem_bytes(n, cl), kvev::select_chunk(n, cl));
    std::printf("cap %d\n", kvev::kSelChunkCap);
    return 0;
}
