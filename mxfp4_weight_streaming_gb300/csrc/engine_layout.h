// Shared-memory plan of one weight-streaming CTA (host and device view).
#pragma once

#include <stdint.h>

namespace mxfp4 {

// Byte offsets inside the 1024-aligned dynamic shared memory of one CTA.
struct SmemLayout {
    uint32_t ring;      // weight ring: nslot stages of steps x BOXES x 2048 bytes
    uint32_t nslot;
    uint32_t steps;     // K steps (256 values) per stage; divides every CTA's steps per unit
    uint32_t group;     // K steps a consumer warp takes at a time (divides steps)
    uint32_t nred;      // partial-sum slots per unit: min(chunks of `group` steps per unit, consumer warps)
    uint32_t xs;        // staged activations, f16 [xcols][blocks][32], column stride xs_stride
    uint32_t fx;        // activation block factors, f32 [4*NT column pairs][blocks][2], stride fx_stride
    uint32_t xs_stride; // bytes per staged column (blocks*64 + 16: the pad spreads columns over banks)
    uint32_t fx_stride; // bytes per column pair of factors (blocks*8 rounded up to 16, + 16)
    uint32_t sc;        // scale ring: nss slots of ss_bytes
    uint32_t nss;
    uint32_t ss_bytes;  // one unit's scales: BOXES x 16 x K/32 bytes
    uint32_t red;       // reduction area: nrb unit buffers x nred_all partial slots (used on cluster rank 0)
    uint32_t nrb;       // units whose partials may be in flight at once
    uint32_t nred_all;  // partial slots per buffer: nred per cluster rank
    uint32_t bars;      // mbarriers: full/empty[nslot], sfull/sempty[nss], staging[5], abort flag
    uint32_t tags;      // u32 words: stage last issued into each ring slot [nslot], unit last
                        // issued into each scale slot [nss], per reduction buffer: item last
                        // finished [nrb], partials handed in [nrb]; per activation buffer:
                        // warps done with it [2], copies issued into it [2]
    // K in parts (part_steps > 0): a CTA walks K in parts of part_steps steps;
    // for each part it streams that part of every unit of a batch of `ubatch`
    // units (one consumer warp each), with the part's activations staged in
    // one of two buffers (xs_buf / fx_buf bytes apart). The reduction area
    // then holds one slot per consumer warp.
    uint32_t part_steps;
    uint32_t ubatch;
    uint32_t xs_buf, fx_buf;
    uint32_t total;
};

// K steps per stage: the largest count <= max_steps / boxes that divides
// every CTA's steps per unit (steps_a and steps_b; 0 counts as divisible).
inline int stage_steps(int boxes, int steps_a, int steps_b, int max_steps = 8) {
    for (int s = max_steps / boxes; s > 1; --s)
        if (steps_a % s == 0 && steps_b % s == 0) return s;
    return 1;
}

// Picks the deepest weight ring (<= 192 KB, >= 2 stages) that fits next to
// the staged activations; the scale ring is deep enough that the producer is
// never held back by it. Returns false if nothing fits.
// nblk is the number of 32-blocks this CTA stages (its part of K); nblk_all
// is the whole row's count (scales cover all of K); steps is the stage size
// and group the consumer chunk (a divisor of steps); unit_steps is the
// largest number of K steps a CTA streams per unit.
// With part_steps > 0 the activations are staged per K part into two
// buffers of nblk blocks each (nblk = the part's blocks), the scale ring has
// ubatch slots (ubatch <= consumer_warps) and the reduction area one slot
// per consumer warp.
inline bool plan_layout(int nt, int boxes, int nblk, int nblk_all, int xcols, int cl, int consumer_warps,
                        int red_stride, int steps, int group, int unit_steps, int max_smem, SmemLayout* out,
                        int part_steps = 0, int ubatch = 0) {
    if (group < 1 || steps % group != 0) return false;
    if (part_steps > 0 && (ubatch < 1 || ubatch > 16 || ubatch > consumer_warps || part_steps % steps != 0 ||
                           group != steps || cl > 1))
        return false;
    const int xbufs = part_steps > 0 ? 2 : 1;
    auto al = [](uint32_t v, uint32_t a) { return (v + a - 1) / a * a; };
    const int nkb = (nblk + 7) / 8;
    const uint32_t slot_bytes = 2048u * boxes * steps;
    const uint32_t xs_stride = static_cast<uint32_t>(nblk) * 64 + 16;
    const uint32_t fx_stride = al(static_cast<uint32_t>(nblk) * 8, 16) + 16;  // 16-byte loads of 2 blocks
    const uint32_t xs_bytes = static_cast<uint32_t>(xcols) * xs_stride;  // one buffer
    const uint32_t fx_bytes = static_cast<uint32_t>(4 * nt) * fx_stride;
    const uint32_t ss_bytes = al(static_cast<uint32_t>(boxes) * 16 * nblk_all, 16);
    int nred = (unit_steps + group - 1) / group;
    nred = nred < 1 ? 1 : (nred > consumer_warps ? consumer_warps : nred);
    if (part_steps > 0) nred = consumer_warps;
    const int ranks = cl > 1 ? cl : 1;
    const uint32_t red_unit_bytes = static_cast<uint32_t>(ranks * nred) * boxes * 8 * nt * red_stride * 4;
    const int budget = max_smem - 1024;
    const int max_slots = static_cast<int>((192u * 1024u) / slot_bytes) < 2 ? 2 : static_cast<int>((192u * 1024u) / slot_bytes);
    // Prefer 4 reduction buffers (owners of 4 consecutive units can hand in
    // their partials without waiting) while the ring keeps >= 4 slots.
    for (int pass = 0; pass < 2; ++pass) {
        const int nrb = part_steps > 0 ? 1 : (pass == 0 ? 4 : 2);
        const uint32_t red_bytes = static_cast<uint32_t>(nrb) * red_unit_bytes;
        for (int nslot = max_slots; nslot >= (pass == 0 ? 4 : 2); --nslot) {
            int nss = (nslot * steps + nkb - 1) / (nkb > 0 ? nkb : 1) + 1;
            nss = nss < 2 ? 2 : (nss > 16 ? 16 : nss);
            if (part_steps > 0) nss = ubatch;  // every unit of a batch keeps its scales for all parts
            SmemLayout l{};
            uint32_t off = 0;
            l.ring = off;
            l.nslot = nslot;
            l.steps = steps;
            l.group = group;
            l.nred = nred;
            off += nslot * slot_bytes;
            l.xs = off;
            l.xs_stride = xs_stride;
            l.xs_buf = xs_bytes;
            off += xbufs * xs_bytes;
            l.fx = off;
            l.fx_stride = fx_stride;
            l.fx_buf = fx_bytes;
            off += xbufs * fx_bytes;
            l.sc = off;
            l.nss = nss;
            l.ss_bytes = ss_bytes;
            off += nss * ss_bytes;
            l.red = off;
            l.nrb = nrb;
            l.nred_all = ranks * nred;
            off += red_bytes;
            l.part_steps = part_steps > 0 ? part_steps : 0;
            l.ubatch = part_steps > 0 ? ubatch : 0;
            l.bars = al(off, 8);
            off = l.bars + 8 * (2 * nslot + 2 * nss + 5 + 1);
            l.tags = off;
            off += 4 * (nslot + nss + 2 * nrb + 4);
            l.total = off;
            if (static_cast<int>(off) <= budget) {
                *out = l;
                return true;
            }
        }
    }
    return false;
}

}  // namespace mxfp4
