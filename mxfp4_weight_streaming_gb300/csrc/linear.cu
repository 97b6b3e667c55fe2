// Weight-streaming MXFP4 linear layer for sm_103a (dense and LM-head shapes).
//
// What it computes ("Zyphra Inference Wave 2", section "Speculative
// decoding"; AMD "megakernel-intro", section "3. Low-Precision Data Types"):
//   y[t][n] = bf16( sum_k x[t][k] * w[n][k] ),  w = e2m1(code) * 2^(s-127)
// for the handful of tokens t of one decode / verify step, reading every
// weight byte from HBM once. A unit is 16 output rows over all of K; the T
// tokens are staged once per CTA (see engine.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "engine.cuh"
#include "linear_launch.h"

namespace mxfp4 {

template <int NT_>
struct DenseProblem {
    static constexpr int NT = NT_;
    static constexpr int BOXES = 1;
    // More consumer warps hide more latency; fewer leave more registers for
    // the wider token tiles.
    static constexpr int NCW = NT == 1 ? 14 : (NT == 2 ? 12 : 8);
    using Params = LinearParams;

    __device__ static int num_units(const Params& p) { return p.n_rg; }
    __device__ static int chunk_of(const Params&, int) { return 0; }
    __device__ static int box_row(const Params&, int u, int) { return u * 16; }
    __device__ static const uint8_t* scale_src(const Params& p, int u, int) {
        return p.ws + (size_t)u * 16 * p.nblk;
    }
    __device__ static int unit_rows(const Params& p, int u) { return min(16, p.N - u * 16); }
    __device__ static int ncols(const Params& p, int) { return p.T; }

    // Staged columns are the T token rows of x (bf16), copied in bulk.
    static constexpr bool kBulkStage = true;
    __device__ static int stage_cols(const Params& p, int) { return p.T; }
    __device__ static const uint8_t* stage_row(const Params& p, int, int col) {
        return reinterpret_cast<const uint8_t*>(p.x + static_cast<size_t>(col) * p.K);
    }

    __device__ static void epilogue(const Params& p, int u, const Sums<NT>& v, int lane) {
        for (int e = lane; e < p.T * 16; e += 32) {
            const int t = e >> 4;
            const int r = e & 15;
            const float s = v.sum(0, t, r);
            const int row = u * 16 + r;
            if (row < p.N) p.y[(size_t)t * p.N + row] = __float2bfloat16_rn(s);
        }
    }
};

static int tokens_to_nt(int T) { return T <= 8 ? 1 : (T <= 16 ? 2 : 4); }

// Plans, in order of preference:
//  1. a lone CTA staging all of K (few_units: at most 4 row groups per SM;
//     whole-stage chunks would then leave most consumer warps idle, so
//     stages are capped at 4 K steps, more and smaller chunks; larger
//     problems keep 7-8 step stages: larger copies, fewer handshakes),
//     when the staged activations leave a ring of at least 64 KB;
//  2. a lone CTA walking K in parts (the activations of all of K do not fit
//     next to such a ring, e.g. T = 16 or 32 at K = 7168), if a CTA holds
//     at least 2 units; else a lone CTA with a smaller ring;
//  3. clusters of 2, 4 or 8 CTAs splitting K (preferred to parts when a CTA
//     would hold a single unit, which parts would re-stage K for alone);
//  4. K in parts whatever the units per CTA.
static bool plan_linear_steps(int T, int K, int max_smem, int max_steps, int max_cl, int units_per_cta, int* cl,
                              SmemLayout* L);
static bool plan_linear_parts(int T, int K, int max_smem, int units_per_cta, SmemLayout* L);

bool plan_linear(int T, int K, int max_smem, bool few_units, int units_per_cta, int* cl, SmemLayout* L) {
    SmemLayout lone{};
    int lone_cl = 1;
    const bool have_lone = (few_units && plan_linear_steps(T, K, max_smem, 4, 1, units_per_cta, &lone_cl, &lone)) ||
                           plan_linear_steps(T, K, max_smem, 8, 1, units_per_cta, &lone_cl, &lone);
    // Whole K per CTA, unless the staged activations leave a ring under
    // 64 KB and parts are an option.
    const bool lone_ring = lone.nslot * lone.steps * 2048u >= 64u * 1024u;
    if (have_lone && (lone_ring || units_per_cta < 2)) {
        *cl = 1;
        *L = lone;
        return true;
    }
    if (units_per_cta >= 2 && plan_linear_parts(T, K, max_smem, units_per_cta, L)) {
        *cl = 1;
        return true;
    }
    if (have_lone) {
        *cl = 1;
        *L = lone;
        return true;
    }
    if (few_units && plan_linear_steps(T, K, max_smem, 4, 8, units_per_cta, cl, L)) return true;
    if (plan_linear_steps(T, K, max_smem, 8, 8, units_per_cta, cl, L)) return true;  // (also when the smaller stages fit no layout)
    *cl = 1;
    return plan_linear_parts(T, K, max_smem, units_per_cta, L);  // last resort for one unit per CTA
}

static int dense_ncw(int nt) {
    return nt == 1 ? DenseProblem<1>::NCW : (nt == 2 ? DenseProblem<2>::NCW : DenseProblem<4>::NCW);
}

static bool plan_linear_steps(int T, int K, int max_smem, int max_steps, int max_cl, int units_per_cta, int* cl,
                              SmemLayout* L) {
    const int nblk = K / 32;
    const int nkb = (K + 255) / 256;
    for (int c = 1; c <= max_cl; c *= 2) {
        if (c > 1 && c > nkb) break;
        const int nkb_c = (nkb + c - 1) / c;
        const int nb_local = nkb_c * 8 < nblk ? nkb_c * 8 : nblk;
        const int nt = tokens_to_nt(T);
        const int ncw = dense_ncw(nt);
        // The stage size must divide the K steps of every rank (the same split
        // the kernel uses: rank r takes [min(nkb, r*nkb_c), min(nkb, +nkb_c))).
        int g = 0;  // gcd of the ranks' step counts (a rank with none adds nothing)
        for (int r = 0; r < c; ++r) {
            const int k0 = r * nkb_c < nkb ? r * nkb_c : nkb;
            const int k1 = k0 + nkb_c < nkb ? k0 + nkb_c : nkb;
            int a = g, b = k1 - k0;
            while (b) {
                const int t = a % b;
                a = b;
                b = t;
            }
            g = a;
        }
        const int steps = stage_steps(1, g, 0, max_steps);
        // Consumer chunk: a whole stage, unless a lone CTA then has fewer
        // chunks than consumer warps (e.g. one row group of 4 steps); then the
        // largest divisor of the stage that gives every warp a chunk, or 1.
        int grp = steps;
        if (c == 1)
            while (grp > 1 && units_per_cta * (nkb / grp) < ncw) {
                int d = grp - 1;
                while (steps % d != 0) --d;
                grp = d;
            }
        if (plan_layout(nt, 1, nb_local, nblk, T, c, ncw, kRedStride, steps, grp, nkb_c, max_smem, L)) {
            *cl = c;
            return true;
        }
    }
    return false;
}

// K in parts: the part (a divisor of the K steps) is the largest whose two
// activation buffers take at most 72 KB; units go in batches of one per
// consumer warp at most (the CTA's share when it fits, halved until the ring
// keeps 64 KB). A stage holds up to 4 K steps of one unit.
static bool plan_linear_parts(int T, int K, int max_smem, int units_per_cta, SmemLayout* L) {
    const int nblk = K / 32;
    const int nkb = (K + 255) / 256;
    const int nt = tokens_to_nt(T);
    const int ncw = dense_ncw(nt);
    int ub_max = units_per_cta < ncw ? units_per_cta : ncw;
    ub_max = ub_max < 16 ? ub_max : 16;
    // First pass: only parts that allow stages of at least 2 steps.
    for (int pass = 0; pass < 2; ++pass) {
        for (int ps = nkb; ps >= 1; --ps) {
            if (nkb % ps != 0) continue;
            if (pass == 0 && ps % 2 != 0 && ps % 3 != 0) continue;
            const int pblk = ps * 8 < nblk ? ps * 8 : nblk;
            if (ps > 1 && 2L * T * (pblk * 64 + 16) > 72L * 1024) continue;
            int spb = 1;
            for (int sb = ps < 4 ? ps : 4; sb >= 1; --sb)
                if (ps % sb == 0) {
                    spb = sb;
                    break;
                }
            for (int ub = ub_max; ub >= 1; ub = ub > 1 ? ub / 2 : 0) {
                // A larger batch re-stages the activations less often, but
                // its scale slots must leave a ring of at least 64 KB.
                if (plan_layout(nt, 1, pblk, nblk, T, 1, ncw, kRedStride, spb, spb, ps, max_smem, L, ps, ub) &&
                    (ub == 1 || L->nslot * L->steps * 2048u >= 64u * 1024u))
                    return true;
            }
        }
    }
    return false;
}

cudaError_t launch_linear(const CUtensorMap& tmap, const LinearParams& p, int num_sms, cudaStream_t stream) {
    const bool parts = p.layout.part_steps != 0;
    switch (tokens_to_nt(p.T)) {
        case 1:
            return parts ? launch_stream_kernel<DenseProblem<1>, true>(tmap, p, p.n_rg, num_sms, stream)
                         : launch_stream_kernel<DenseProblem<1>>(tmap, p, p.n_rg, num_sms, stream);
        case 2:
            return parts ? launch_stream_kernel<DenseProblem<2>, true>(tmap, p, p.n_rg, num_sms, stream)
                         : launch_stream_kernel<DenseProblem<2>>(tmap, p, p.n_rg, num_sms, stream);
        default:
            return parts ? launch_stream_kernel<DenseProblem<4>, true>(tmap, p, p.n_rg, num_sms, stream)
                         : launch_stream_kernel<DenseProblem<4>>(tmap, p, p.n_rg, num_sms, stream);
    }
}

}  // namespace mxfp4
