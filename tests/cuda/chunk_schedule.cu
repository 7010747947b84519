// Host-only check of the codec kernels' order of chunks (cta_chunks in spl_device.cuh and
// wave_grid in spl_kernels.h): for each (chunks, resident CTAs, chunks per CTA) case, the CTAs
// of the grid the launchers use take every chunk exactly once, each CTA's chunks lie in its
// own wave, and no CTA takes more than its chunks per CTA.  Runs on the CPU; prints one line
// per failing case and exits nonzero if any fails.  Built and run by the CPU tests.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "spl_device.cuh"
#include "spl_kernels.h"

int main() {
    const int64_t totals[] = {1, 2, 5, 151, 152, 607, 608, 609, 1000, 1216, 4863, 9727, 9728,
                              9729, 19456, 40000, 262143, 262144, 262145, 300001};
    const int residents[] = {1, 7, 152, 304, 608, 1216};
    const int per_ctas[] = {1, 3, 8, 16, 32, 64, spl::kSendChunksPerCta, spl::kRecvChunksPerCta};
    int failures = 0;
    int64_t cases = 0;
    for (int64_t total : totals) {
        for (int resident : residents) {
            for (int per_cta : per_ctas) {
                ++cases;
                const int grid = spl::wave_grid(total, resident, per_cta);
                std::vector<int> seen(static_cast<size_t>(total), 0);
                bool ok = grid >= 1;
                for (int64_t b = 0; b < grid && ok; ++b) {
                    const spl::ChunkSpan s = spl::cta_chunks(total, resident, per_cta, b);
                    const int64_t wave = b / resident;
                    const int64_t lo = wave * resident * per_cta;
                    int taken = 0;
                    for (int64_t c = s.first; c < s.end; c += resident) {
                        if (c < lo || c >= lo + static_cast<int64_t>(resident) * per_cta ||
                            c >= total) {
                            ok = false;
                            break;
                        }
                        ++seen[static_cast<size_t>(c)];
                        ++taken;
                    }
                    if (taken > per_cta) ok = false;
                }
                for (int64_t c = 0; c < total && ok; ++c)
                    if (seen[static_cast<size_t>(c)] != 1) ok = false;
                if (!ok) {
                    std::printf("FAIL total=%lld resident=%d per_cta=%d grid=%d\n",
                                static_cast<long long>(total), resident, per_cta, grid);
                    ++failures;
                }
            }
        }
    }
    std::printf("%lld cases, %d failed\n", static_cast<long long>(cases), failures);
    return failures == 0 ? 0 : 1;
}
