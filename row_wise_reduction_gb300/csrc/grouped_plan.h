// Launch plan of the row-group split-row softmax (split_grouped_kernel in
// online_softmax_persistent.cuh) [Triton Kernel 实现练习 §2.5
// split_online_softmax]: how many CTAs share a row, how large their slices
// and ring buffers are, and how many CTAs the cooperative grid has. Pure host
// arithmetic (no CUDA call), so that it is tested on the CPU.
#pragma once

#include <cstdint>

namespace rowops {

constexpr int kGroupedMaxBuffers = 8;  // ring buffers per CTA, at most
constexpr int kGroupedMaxVpt = 7;      // vectors of a slice per thread (slices of at most block * 7 vectors)
constexpr int kGroupedMaxSlots = 160;  // CTAs per row group, at most (a multiple of 32)

struct GroupedLimits {
    int block;              // threads per CTA
    int per_sm;             // CTAs per SM
    int max_vpt;            // 16-byte vectors of a slice per thread (held in registers)
    int max_slots;          // CTAs per row group, at most
    int max_buffers;        // ring buffers per CTA, at most
    int64_t ring_bytes;     // shared memory a CTA's ring may take
};

struct GroupedPlan {
    int n = 0;              // CTAs per row group; 0: the form does not apply
    int64_t slot_vecs = 0;  // 16-byte vectors per ring buffer (>= the widest slice, a multiple of 8)
    int nbuf = 0;           // ring buffers per CTA
    int64_t grid = 0;       // CTAs of the grid: rows per wave x n
};

// M rows of nvec 16-byte vectors on num_sms SMs. n is the smallest divisor of
// the grid's CTA slots (num_sms x per_sm) whose slices (ceil(nvec / n)
// vectors) fit the block's registers and min_buffers (at least 2) ring
// buffers, raised to the next divisor while M * n is below the CTA slots, so
// that few rows still cover every SM; then the ring takes as many slices as
// fit, up to max_buffers. Not applicable (n = 0) when no divisor fits, when n
// would exceed max_slots or slots_per_row (the workspace's slots per row), or
// when a slice would hold fewer than 32 vectors.
inline GroupedPlan grouped_plan(int64_t M, int64_t nvec, int num_sms, int min_buffers, int64_t slots_per_row,
                                const GroupedLimits& lim) {
    GroupedPlan p;
    if (M < 1 || nvec < 1 || num_sms < 1 || lim.per_sm < 1) return p;
    const int ctas = num_sms * lim.per_sm;
    const int want = min_buffers >= 2 ? min_buffers : 2;
    auto slot_vecs_for = [&](int d) { return ((nvec + d - 1) / d + 7) / 8 * 8; };
    auto fits = [&](int d) {
        return (nvec + d - 1) / d <= int64_t(lim.block) * lim.max_vpt && slot_vecs_for(d) * 16 * want <= lim.ring_bytes;
    };
    int n = 0;
    for (int d = 1; d <= ctas && n == 0; ++d)
        if (ctas % d == 0 && fits(d)) n = d;
    if (n == 0) return p;
    while (M * n < ctas && n < ctas) {
        int d = n + 1;
        while (ctas % d != 0) ++d;
        n = d;
    }
    if (n > lim.max_slots || nvec < int64_t(n) * 32 || n > slots_per_row) return p;
    p.n = n;
    p.slot_vecs = slot_vecs_for(n);
    const int64_t nbuf = lim.ring_bytes / (p.slot_vecs * 16);
    p.nbuf = int(nbuf > lim.max_buffers ? lim.max_buffers : nbuf);
    const int64_t rows_per_wave = (ctas / n) < M ? (ctas / n) : M;
    p.grid = rows_per_wave * n;
    return p;
}

}  // namespace rowops
