// Host entry point over the workqueue's balance-order map (plan_map.cuh), so
// that a CPU test can check the map the self-planning decode uses against an
// enumeration of the plan.  Built by tests/test_plan_map.py into a temporary
// directory.
#include "plan_map.cuh"

extern "C" int plan_map_all(int B, const int *F, const int *R, const int16_t *S, int Hkv, int Hq,
                            int G, int T, int *rec, long long *lex)
{
    for (int t = 0; t < T; ++t) {
        int64_t k = -1;
        const int4 r = pkv::plan_task_at(t, F, R, S, B, Hkv, Hq, G, &k);
        rec[4 * t] = r.x;
        rec[4 * t + 1] = r.y;
        rec[4 * t + 2] = r.z;
        rec[4 * t + 3] = r.w;
        lex[t] = k;
    }
    return 0;
}
