// Host-side check of the tensor-core projection's launch plan (plan_projection and
// choose_chunks in tc_common.cuh) over a sweep of shapes: every plan must give
// non-empty chunks that cover the sequence, a shared-memory ring that fits the SM and
// leaves room for the split reduction's two 32 KB slices, pairs only where the kernel
// supports them, the TMEM columns of the CTAs resident on one SM within 512, and
// split partials within the budget.  Prints the number of plans checked, or the
// first violated property, and returns non-zero on a violation.
#include <cstdio>

#include "../../rank_linear_complexity_gb300/csrc/tc_common.cuh"

using namespace linformer::tc;

static int fail(const char *what, int n, long long members, long long groups, int mh, int dist,
                int ragged, int sms, size_t budget) {
    std::printf("FAIL %s: n=%d members=%lld groups=%lld mhalves=%d distinct=%d ragged=%d sms=%d "
                "budget=%zu\n", what, n, members, groups, mh, dist, ragged, sms, budget);
    return 1;
}

int main() {
    const int ns[] = {8, 64, 200, 256, 320, 512, 777, 1000, 4096, 6144, 6200, 16384, 65536, 131072};
    const long long members_list[] = {1, 2, 3, 8, 16, 32, 100, 152, 304, 1000};
    const long long groups_list[] = {1, 2, 12, 16};
    const int sms_list[] = {148, 152};
    const size_t budgets[] = {~size_t(0), size_t(32) << 20, size_t(1) << 20, 0};
    long long checked = 0;
    for (int n : ns)
        for (long long members : members_list)
            for (long long groups : groups_list)
                for (int mh = 1; mh <= 2; ++mh)
                    for (int dist = 0; dist <= 1; ++dist)
                        for (int ragged = 0; ragged <= 1; ++ragged)
                            for (int sms : sms_list)
                                for (size_t budget : budgets) {
#define CHECK(cond, what) \
    if (!(cond)) return fail(what, n, members, groups, mh, dist, ragged, sms, budget)
        const ProjPlan p = plan_projection(n, members, groups, mh, dist, ragged != 0, sms, budget);
        const long long units = members * groups;
        CHECK(p.C >= 1 && p.C <= 64, "chunk count in [1, 64]");
        CHECK(p.C == 1 || p.C <= n / 256, "at least 256 rows a chunk when split");
        CHECK(p.CH % kBK == 0 && p.CH > 0, "chunk rows a multiple of the stage");
        CHECK((long long)p.C * p.CH >= n && (long long)(p.C - 1) * p.CH < n,
              "chunks cover the sequence and none is empty");
        CHECK(partial_bytes(units, p.C, mh) <= budget || p.C == 1, "partials within budget");
        CHECK(p.stages >= 2 && p.stages <= 6, "ring depth in [2, 6]");
        CHECK(p.smem <= 227 * 1024, "shared memory within one CTA's limit");
        CHECK(p.smem >= 1024 + kProjectMinRing + 256, "ring holds the reduction's slices and staging");
        CHECK(p.threads != 256 || p.smem >= 1024 + kProjectMinRingWide + 256,
              "eight-warp launches: ring holds both groups' staging buffers");
        CHECK(p.smem >= 1024 + project_stage_bytes(mh, dist, 1) * p.stages + 256,
              "one-unit ring fits");
        CHECK(p.pairs >= 0 && p.pairs <= members / 2, "at most members / 2 pairs");
        if (p.pairs > 0) {
            CHECK(p.C == 1 && !dist && !ragged, "pairs only unsplit, E = F, no lengths");
            CHECK(p.stages2 >= 2 && p.stages2 <= 6, "pair ring depth in [2, 6]");
            CHECK(p.smem >= 1024 + project_stage_bytes(mh, 0, 2) * p.stages2 + 256,
                  "two-unit ring fits");
        }
        CHECK(p.threads == ((p.pairs > 0 && mh == 2) ? 256 : 128), "thread count");
        CHECK(p.grid == groups * p.C * (members - p.pairs) && p.grid >= 1, "grid size");
        // TMEM: a CTA holds mhalves x (1 or 2 units) x 128 columns; the CTAs resident on
        // one SM must fit in 512 or an allocation would wait for another CTA to exit.
        const int ctas = project_ctas_per_sm(p.smem);
        const int cols = mh * (p.pairs > 0 ? 2 : 1) * 128;
        CHECK(ctas * cols <= 512, "TMEM columns of co-resident CTAs within 512");
        ++checked;
                                }
    std::printf("ok %lld plans\n", checked);
    return 0;
}
