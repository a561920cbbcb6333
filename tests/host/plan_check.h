// Shared part of the launch-planner host checks (plan_check_pn.cu, plan_check_nvfp4.cu): the
// shared-memory layout of one accepted plan, checked against the regions the kernel's accessors
// use. Host code only; included after the translation unit whose planner is checked.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

namespace plan_check {

int failures = 0;
long plans = 0;

struct Region {
    uint64_t lo, hi;
    const char* name;
};

// What the kernel reads and writes besides the plan's offsets.
struct Shape {
    int M;
    uint64_t slot_need;      // bytes of one operand slot the kernel uses
    uint64_t x_unit_bytes;   // resident: x bytes per (unit, activation row)
    uint64_t x_buf_bytes;    // streaming: bytes of one x buffer
    uint64_t stage_bytes;    // one weight stage
    bool stage_1024;         // the stages need 1024-byte alignment (128-byte swizzled copies)
};

#define PC_FAIL(...)                                                                             \
    do {                                                                                         \
        if (plan_check::failures++ < 5) {                                                        \
            std::printf("FAIL %s: ", what);                                                      \
            std::printf(__VA_ARGS__);                                                            \
            std::printf("\n");                                                                   \
        }                                                                                        \
        return;                                                                                  \
    } while (0)

template <class P>
void check_plan(const P& p, const Shape& s, uint64_t smem_limit, uint32_t resident_flag, uint32_t overlap_flag,
                int part_pitch, const char* what) {
    ++plans;
    const auto& sc = p.sc;
    if (sc.G < 1 || sc.G > sc.items) PC_FAIL("grid %d for %d items", sc.G, sc.items);
    if (p.NS < 2) PC_FAIL("%d weight stages", p.NS);
    if (p.total + 1024ull > smem_limit) PC_FAIL("total %u + 1024 over the limit", p.total);
    // largest share, span of any share, and whether some tile is shared by two CTAs
    int most = 0, span = 0;
    bool shared = !sc.tile_major && sc.U > 1;
    for (int c = 0; c < sc.G; ++c) {
        const int i0 = sc.first(c), i1 = sc.first(c + 1);
        most = std::max(most, i1 - i0);
        span = std::max(span, sc.span(i0, i1));
        if (c > 0 && sc.tile_of(i0) == sc.tile_of(i0 - 1)) shared = true;
    }
    if (p.list_cap < most) PC_FAIL("list capacity %d below a share of %d items", p.list_cap, most);
    if (p.publish != shared) PC_FAIL("publish %d but tiles shared %d", p.publish, shared);
    if (p.slot_bytes < s.slot_need || p.slot_bytes % 128) PC_FAIL("slot of %u bytes, need %llu", p.slot_bytes,
                                                                    (unsigned long long)s.slot_need);
    if (p.part_off % 16 || p.list_off % 16 || p.ring_off % 128 || p.xs_off % 16)
        PC_FAIL("misaligned region: list %u part %u ring %u xs %u", p.list_off, p.part_off, p.ring_off, p.xs_off);
    if (p.stage_off % (s.stage_1024 ? 1024 : 128)) PC_FAIL("stages at %u", p.stage_off);
    const bool resident = (p.mode & resident_flag) != 0, overlap = (p.mode & overlap_flag) != 0;
    const uint64_t stages_end = p.stage_off + static_cast<uint64_t>(p.NS) * s.stage_bytes;
    if (stages_end != p.total) PC_FAIL("stages end at %llu, total %u", (unsigned long long)stages_end, p.total);
    std::vector<Region> r;
    r.push_back({0, 8ull * (2 * p.NS + 2 * p.RB + 5), "barriers"});
    r.push_back({p.list_off, p.list_off + 4ull * (4 + 2ull * p.list_cap), "lists"});
    r.push_back({p.part_off, p.part_off + 4ull * 4 * s.M * part_pitch, "row sums"});
    uint64_t x_lo = p.xs_off, x_hi;
    if (resident) {
        if (p.RB != 0) PC_FAIL("resident plan with %d ring slots", p.RB);
        x_hi = x_lo + static_cast<uint64_t>(span) * s.M * s.x_unit_bytes;
        r.push_back({p.ring_off, p.ring_off + static_cast<uint64_t>(span) * p.slot_bytes, "operand slots"});
        if (overlap) {
            const uint64_t first = p.stage_off + static_cast<uint64_t>(p.x_stage) * s.stage_bytes;
            if (p.x_stage < 0 || p.x_stage >= p.NS || x_lo != first || x_hi > p.total)
                PC_FAIL("x in stages %d.. of %d: [%llu, %llu) total %u", p.x_stage, p.NS, (unsigned long long)x_lo,
                        (unsigned long long)x_hi, p.total);
        } else {
            if (p.x_stage != p.NS) PC_FAIL("x stage %d without overlap", p.x_stage);
            r.push_back({x_lo, x_hi, "x"});
        }
    } else {
        if (p.RB < 2 || p.XB < 1) PC_FAIL("streaming plan with %d slots, %d x buffers", p.RB, p.XB);
        x_hi = x_lo + static_cast<uint64_t>(p.XB) * s.x_buf_bytes;
        r.push_back({x_lo, x_hi, "x"});
        r.push_back({p.ring_off, p.ring_off + static_cast<uint64_t>(p.RB) * p.slot_bytes, "operand slots"});
    }
    r.push_back({p.stage_off, stages_end, "stages"});
    std::sort(r.begin(), r.end(), [](const Region& a, const Region& b) { return a.lo < b.lo; });
    for (size_t k = 1; k < r.size(); ++k)
        if (r[k].lo < r[k - 1].hi)
            PC_FAIL("%s [%llu, %llu) overlaps %s [%llu, %llu)", r[k].name, (unsigned long long)r[k].lo,
                    (unsigned long long)r[k].hi, r[k - 1].name, (unsigned long long)r[k - 1].lo,
                    (unsigned long long)r[k - 1].hi);
}

}  // namespace plan_check
