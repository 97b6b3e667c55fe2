// The weight-streaming engine shared by the dense / LM-head linear kernel and
// the two MoE expert kernels.
//
// A kernel streams a sequence of "units". A unit is one group of 16 weight
// rows (or BOXES groups of 16 rows that share their activations, e.g. the
// gate and up rows of one expert) over the whole reduction dimension K,
// applied to a small set of activation columns (tokens). Consecutive units
// with the same activation columns form a "chunk"; the activations of a
// chunk are staged once into shared memory.
//
// One persistent CTA per SM (or per cluster rank), warp-specialised:
//   producer warp : per unit, one bulk copy of the scale bytes of each row
//                   group (16 rows x K/32 contiguous bytes) into a scale
//                   ring; per stage (spb K steps of 256 values), one TMA
//                   copy per box of 16 rows x spb 128-byte segments
//                   (SWIZZLE_128B) into a ring slot, which it tags with the
//                   stage index.
//   consumer warps: the K steps are cut into chunks of G steps, dealt
//                   round-robin over the warps. Per 32-value block: ldmatrix
//                   -> hardware E2M1 -> f16 unpack -> two m16n8k16 MMAs
//                   (fp32 accumulate) per 8-column tile -> partial scaled by
//                   2^(s-127) * column factor (f32x2) into the accumulators.
//                   Per unit, each owning warp hands its partial to a
//                   reduction buffer; one owner sums the partials in a fixed
//                   order and runs the problem's epilogue (deterministic).
// K in parts (stream_kernel<P, true>, dense problem): when the activations
// of all of K do not fit, a lone CTA walks K in parts with double-buffered
// activation parts, and each unit of a batch stays with one consumer warp,
// its sums in registers, across all parts.
// Every wait is bounded (see device_common.cuh); on a timeout the kernel
// records it in the status word and winds down.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "device_common.cuh"
#include "engine_layout.h"

namespace mxfp4 {

// Whether a problem gates its staging on inputs that other CTAs produce
// (P::kInputGate and P::wait_inputs).
template <class P, class = void>
struct HasInputGate : std::false_type {};
template <class P>
struct HasInputGate<P, std::void_t<decltype(P::kInputGate)>> : std::bool_constant<P::kInputGate> {};

// Warps of a CTA: P::NCW consumers, then the producer.
template <class P>
struct Roles {
    static constexpr int kConsumers = P::NCW;
    static constexpr int kProducer = P::NCW;
    static constexpr int kThreads = (P::NCW + 1) * 32;
    static constexpr int kConsumerThreads = P::NCW * 32;
};
constexpr int kBoxBytes = 2048;  // 16 rows x 128 bytes = 16 rows x 256 K values

// How the producer copies a stage (Params::tma3d):
//   0: 2D map [rows, K/2 B], one 16-row x 128-byte box per step and box;
//   1: 3D map (128 B, rows, K/256), one copy per box of 16 rows x spb steps;
//   kCopyMerged3d: 3D map whose box is 16 * BOXES rows high, the boxes of a
//      unit being consecutive rows: one copy per stage;
//   kCopyMerged5d: 5D map (128 B, 16 rows, box, 16-row group, K/256) whose
//      box-index stride is the distance between a unit's boxes (the gate and
//      up rows of an expert): one copy per stage.
// The merged copies land a stage as [step][box][16 rows][128 B].
constexpr int kCopyMerged3d = 2;
constexpr int kCopyMerged5d = 3;

__device__ __forceinline__ void issue_merged_stage(int mode, uint32_t dst, const CUtensorMap* tmap, int row0, int kb,
                                                   uint32_t bar, uint64_t policy) {
    if (mode == kCopyMerged3d)
        tma_load_3d(dst, tmap, 0, row0, kb, bar, policy);
    else
        tma_load_5d(dst, tmap, 0, 0, 0, row0 / 16, kb, bar, policy);
}
constexpr int kRedStride = 20;   // floats per column row of the reduction area (16 + 4 pad)

// mbarriers and tag words of one CTA (shared addresses), in the order the
// layout plans them.
struct Bars {
    uint32_t base;
    uint32_t nslot, nss, nrb;
    uint32_t tags;
    __device__ uint32_t full(uint32_t s) const { return base + 8 * s; }
    __device__ uint32_t empty(uint32_t s) const { return base + 8 * (nslot + s); }
    __device__ uint32_t sfull(uint32_t s) const { return base + 8 * (2 * nslot + s); }
    __device__ uint32_t sempty(uint32_t s) const { return base + 8 * (2 * nslot + nss + s); }
    // Whole-K staging: xbar(0), xbar(1): all consumers before / after
    // staging; xbar(2): the bulk copies of raw activations have landed.
    // K in parts: xbar(b) (b = 0, 1): the raw activations of a part have
    // landed in buffer b; xbar(2 + b): every consumer has converted its
    // share of buffer b.
    __device__ uint32_t xbar(uint32_t b) const { return base + 8 * (2 * nslot + 2 * nss + b); }
    __device__ uint32_t abort_flag() const { return base + 8 * (2 * nslot + 2 * nss + 5); }
    // Stage last issued into ring slot s; unit last issued into scale slot s.
    __device__ uint32_t ring_tag(uint32_t s) const { return tags + 4 * s; }
    __device__ uint32_t scale_tag(uint32_t s) const { return tags + 4 * (nslot + s); }
    // Per reduction buffer: unit whose partials it last held (a copy on
    // every cluster rank), and how many owners have handed in theirs (the
    // count on rank 0 is the one used).
    __device__ uint32_t red_tag(uint32_t b) const { return tags + 4 * (nslot + nss + b); }
    __device__ uint32_t red_count(uint32_t b) const { return tags + 4 * (nslot + nss + nrb + b); }
    // K in parts: consumer warps that have left the part in buffer b.
    __device__ uint32_t xdone(uint32_t b) const { return tags + 4 * (nslot + nss + 2 * nrb + b); }
    // K in parts: copies issued into buffer b so far.
    __device__ uint32_t xissued(uint32_t b) const { return tags + 4 * (nslot + nss + 2 * nrb + 2 + b); }
};

// Next position of a ring of n slots: slot index and the parity of its
// current round (no division on the per-unit path).
__device__ __forceinline__ void ring_next(uint32_t& i, uint32_t& phase, uint32_t n) {
    if (++i == n) {
        i = 0;
        phase ^= 1u;
    }
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtx& w) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, w));
}

// ------------------------------------------------------------------------
// Activation staging helpers (used by the problems' stage()).
//
// A column is 32 values of one 32-block stored as f16 = v * 2^c, c chosen
// per (column, block) so the block's largest magnitude lands in [2^14,
// 2^15); the factor 2^-c goes to fx. Multiplying by a power of two is exact,
// and a bf16 value (8 significant bits) is exact in f16 when the result is
// at least 2^-17, i.e. for every element within 2^31 of its block maximum.

// Where a problem's stage() writes: column c of 32-block b (relative to the
// CTA's first block) and its factor. Columns are 16 bytes apart in bank
// terms (stride = blocks*64 + 16) so the 8 columns a warp reads per block
// hit different banks; factors sit in column pairs [pair][block][2].
struct StageDst {
    uint8_t* xs;
    uint8_t* fx;
    uint32_t xs_stride, fx_stride;
    // Set to 1 when a staged block gets a factor above 1 (its largest
    // magnitude is at least 2^15): only then can a weight scale times the
    // factor exceed float range, and the consumers switch to the wide path.
    volatile int* wide;
    __device__ uint8_t* col(int c, int b) const { return xs + c * xs_stride + b * 64; }
    __device__ float* factor(int c, int b) const {
        return reinterpret_cast<float*>(fx + (c >> 1) * fx_stride + b * 8 + (c & 1) * 4);
    }
};

// Floor of log2 of a positive float given its bit pattern (no sign).
__device__ __forceinline__ int floor_log2_f32_bits(uint32_t a) {
    const int e = static_cast<int>(a >> 23);
    return e ? e - 127 : (31 - __clz(static_cast<int>(a))) - 149;
}

// Scale exponent c for a block whose largest |value| has floor(log2) fl
// (capped so the factor 2^-c stays a representable float).
__device__ __forceinline__ int staging_exponent(int fl) { return min(14 - fl, 149); }

// v * 2^c for c in [-149 + 14, 149 + 14] without overflow in the factor.
struct Pow2Scaler {
    float s1, s2;
    bool two;
    __device__ explicit Pow2Scaler(int c) {
        two = c > 127 || c < -126;
        const int c1 = two ? (c > 0 ? 64 : -64) : 0;
        s1 = exp2_int(c - c1);
        s2 = exp2_int(c1);
    }
    __device__ float operator()(float v) const { return two ? (v * s1) * s2 : v * s1; }
};

// Stage one block of 32 bf16 values (16 words) as f16 column data.
__device__ __forceinline__ void stage_bf16_block(const uint32_t (&w)[16], uint8_t* dst, float* fx_out,
                                                 volatile int* wide) {
    // Largest magnitude: a depth-4 tree of packed 16-bit maxima.
    uint32_t m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = __vmaxu2(w[2 * j] & 0x7fff7fffu, w[2 * j + 1] & 0x7fff7fffu);
#pragma unroll
    for (int j = 0; j < 4; ++j) m[j] = __vmaxu2(m[j], m[j + 4]);
    m[0] = __vmaxu2(__vmaxu2(m[0], m[2]), __vmaxu2(m[1], m[3]));
    const uint32_t amax = max(m[0] & 0xffffu, m[0] >> 16);
    int c = 0;
    if (amax != 0) c = staging_exponent(floor_log2_f32_bits(amax << 16));
    if (c < 0) *wide = 1;
    const Pow2Scaler sc(c);
    uint32_t o[16];
    if (!sc.two) {
        // One packed multiply per pair of values (the usual case).
        const uint64_t s2 = f32x2_pack(sc.s1, sc.s1);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 v = f32x2_unpack(
                f32x2_mul(f32x2_pack(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u)), s2));
            __half2 h = __floats2half2_rn(v.x, v.y);
            o[j] = *reinterpret_cast<uint32_t*>(&h);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            __half2 h = __floats2half2_rn(sc(__uint_as_float(w[j] << 16)), sc(__uint_as_float(w[j] & 0xffff0000u)));
            o[j] = *reinterpret_cast<uint32_t*>(&h);
        }
    }
    const uint32_t d = smem_addr(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) sts128(d + 16 * q, o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    *fx_out = exp2_int(-c);
}

// Stage one block of 32 fp32 values as an exact-to-22-bits pair of f16
// columns: hi = f16(v * 2^c), lo = f16(v * 2^c - hi). Both share the factor.
__device__ __forceinline__ void stage_f32_block_split(const float (&v)[32], uint8_t* dst_hi, uint8_t* dst_lo,
                                                      float* fx_hi, float* fx_lo, volatile int* wide) {
    uint32_t amax = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = max(amax, __float_as_uint(v[j]) & 0x7fffffffu);
    int c = 0;
    if (amax != 0) c = staging_exponent(floor_log2_f32_bits(amax));
    if (c < 0) *wide = 1;
    const Pow2Scaler sc(c);
    uint32_t oh[16], ol[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float a = sc(v[2 * j]);
        const float b = sc(v[2 * j + 1]);
        const __half2 hi = __floats2half2_rn(a, b);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(a - hf.x, b - hf.y);
        oh[j] = *reinterpret_cast<const uint32_t*>(&hi);
        ol[j] = *reinterpret_cast<const uint32_t*>(&lo);
    }
    uint4* dh = reinterpret_cast<uint4*>(dst_hi);
    uint4* dl = reinterpret_cast<uint4*>(dst_lo);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        dh[q] = make_uint4(oh[4 * q], oh[4 * q + 1], oh[4 * q + 2], oh[4 * q + 3]);
        dl[q] = make_uint4(ol[4 * q], ol[4 * q + 1], ol[4 * q + 2], ol[4 * q + 3]);
    }
    const float f = exp2_int(-c);
    *fx_hi = f;
    *fx_lo = f;
}

// ------------------------------------------------------------------------
// Activation staging by bulk copy: for problems whose staged columns are
// bf16 rows of K values (P::kBulkStage), one thread copies each column's
// K range [kblk0*32, kblk1*32) straight into its staged column (the byte
// layout is the same: 64 bytes per 32-block), then every consumer thread
// converts blocks in place. Only shared-memory latency is on the path,
// instead of one dependent global load per block and thread.

// One thread: the copies of a chunk's columns into the columns at xs_s,
// completing on the transaction barrier xfull.
template <class P>
__device__ __forceinline__ void issue_column_copies(const typename P::Params& p, int chunk, int kblk0, int kblk1,
                                                    uint32_t xs_s, uint32_t xs_stride, uint32_t xfull) {
    const int ncol = P::stage_cols(p, chunk);
    const int nb = kblk1 - kblk0;
    fence_proxy_async_shared();  // earlier reads / writes of the columns come first
    mbar_arrive_expect_tx(xfull, static_cast<uint32_t>(ncol * nb * 64));
    if (nb > 0)
        for (int t = 0; t < ncol; ++t)
            bulk_load_plain(xs_s + t * xs_stride, P::stage_row(p, chunk, t) + static_cast<size_t>(kblk0) * 64,
                            static_cast<uint32_t>(nb * 64), xfull);
}

// Thread tid of nthreads: converts its share of the landed bf16 blocks of
// ncol columns (nb blocks each) in place, and zeroes the factors of the
// tile's unused columns (kCols = 8 * NT).
template <int kCols>
__device__ __forceinline__ void convert_columns(int ncol, int nb, const StageDst& dst, uint32_t xs_s, int tid,
                                                int nthreads) {
    // Consecutive threads take consecutive columns of one block: the padded
    // column stride puts them 4 banks apart, so a warp's 16-byte accesses
    // need 4 wavefronts for T >= 4 (consecutive blocks of one column, 64
    // bytes apart, would need 16).
    // Item it = b * ncol + t, advanced by nthreads without a division.
    const int db = nthreads / ncol, dt = nthreads - db * ncol;
    int b = tid / ncol, t = tid - (tid / ncol) * ncol;
    for (int it = tid; it < ncol * nb; it += nthreads) {
        const uint32_t a = xs_s + t * dst.xs_stride + b * 64;
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = lds128(a + 16 * q);
            w[4 * q] = v.x;
            w[4 * q + 1] = v.y;
            w[4 * q + 2] = v.z;
            w[4 * q + 3] = v.w;
        }
        stage_bf16_block(w, dst.col(t, b), dst.factor(t, b), dst.wide);
        t += dt;
        b += db;
        if (t >= ncol) {
            t -= ncol;
            ++b;
        }
    }
    const int nz = kCols - ncol;
    if (nz > 0) {
        const int zb = nthreads / nz, zt = nthreads - zb * nz;
        int bz = tid / nz, tz = tid - (tid / nz) * nz;
        for (int it = tid; it < nb * nz; it += nthreads) {
            *dst.factor(ncol + tz, bz) = 0.0f;
            tz += zt;
            bz += zb;
            if (tz >= nz) {
                tz -= nz;
                ++bz;
            }
        }
    }
}

// Whole-K staging of one chunk: copy, wait, convert (all consumer threads).
template <class P>
__device__ __forceinline__ bool stage_bulk(const typename P::Params& p, int chunk, int kblk0, int kblk1,
                                           const StageDst& dst, uint32_t xs_s, uint32_t xfull, uint32_t parity,
                                           const WaitCtx& wc, int tid, int nthreads) {
    if (tid == 0) issue_column_copies<P>(p, chunk, kblk0, kblk1, xs_s, dst.xs_stride, xfull);
    if (!__all_sync(0xffffffffu, mbar_wait(xfull, parity, wc))) return false;
    convert_columns<8 * P::NT>(P::stage_cols(p, chunk), kblk1 - kblk0, dst, xs_s, tid, nthreads);
    return true;
}

// ------------------------------------------------------------------------
// One K step of one unit: BOXES boxes of 16 rows x 256 K (8 blocks of 32;
// fewer at the end of K), against the staged columns. Blocks are numbered
// globally (scales) and relative to kblk0 (staged activations).
//
// Per block, the two MMAs give the exact-product sums d of the unscaled
// codes and staged activations; the block's weight scale (per row) times
// its activation factor (per column) is a power of two, and the pair
// {d0, d1} (one row, two columns) is scaled and accumulated with one f32x2
// multiply and one f32x2 FMA. acc[bx][n] = {{row g: col 2t, 2t+1}, {row g+8:
// col 2t, 2t+1}} of n-tile n.
// kWide: the weight scale and the activation factor are applied one after
// the other in double precision, so no intermediate leaves float range
// unless the result does (the CTA staged a block with a factor above 1).
template <int NT, int BOXES, bool kWide = false>
__device__ __forceinline__ void consume_step(uint32_t slot, uint32_t box_stride, uint32_t sc, int nblk, int kb,
                                             int kblk0, int kblk1, int ncols, uint32_t xs, uint32_t xs_stride,
                                             uint32_t fx, uint32_t fx_stride, uint64_t (&acc)[BOXES][NT][2],
                                             int lane) {
    const int g = lane >> 2;
    const int tig = lane & 3;
    const int mi = lane >> 3;
    const int row = ((mi & 1) << 3) | (lane & 7);
    const int bsel = mi >> 1;
#pragma unroll
    for (int jp = 0; jp < 4; ++jp) {
        const int b_first = kb * 8 + 2 * jp;
        if (b_first >= kblk1) break;
        const uint32_t roff = row * 128 + (((2 * jp + bsel) ^ (row & 7)) << 4);
        uint32_t r[BOXES][4];
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx)
            ldmatrix_x4(slot + bx * box_stride + roff, r[bx][0], r[bx][1], r[bx][2], r[bx][3]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int b = b_first + h;
            if (b >= kblk1) break;
            const int bl = b - kblk0;
            uint4 xv[NT];
            uint64_t F[NT];
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int col = min(g + 8 * n, ncols - 1);  // see consume_step_full
                xv[n] = lds128(xs + col * xs_stride + bl * 64 + tig * 16);
                F[n] = lds64_pair(fx + (tig + 4 * n) * fx_stride + bl * 8);
            }
#pragma unroll
            for (int bx = 0; bx < BOXES; ++bx) {
                const uint32_t scb = sc + bx * 16 * nblk + b;
                const uint32_t fw = e8m0x2_to_bf16x2(lds_u8(scb + g * nblk) | (lds_u8(scb + (g + 8) * nblk) << 8));
                const float fw0 = __uint_as_float(fw << 16), fw1 = __uint_as_float(fw & 0xffff0000u);
                const uint64_t W0 = f32x2_pack(fw0, fw0), W1 = f32x2_pack(fw1, fw1);
                uint32_t ga[4], gb[4];
                e2m1x8_to_f16x8(r[bx][2 * h], ga[0], ga[1], ga[2], ga[3]);
                e2m1x8_to_f16x8(r[bx][2 * h + 1], gb[0], gb[1], gb[2], gb[3]);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    uint64_t d01, d23;
                    mma_f16_k32(d01, d23, ga, gb, xv[n]);
                    if constexpr (kWide) {
                        const float2 f = f32x2_unpack(F[n]);
                        const float2 a = f32x2_unpack(d01), c = f32x2_unpack(d23);
                        float2 s0 = f32x2_unpack(acc[bx][n][0]), s1 = f32x2_unpack(acc[bx][n][1]);
                        s0.x += static_cast<float>(static_cast<double>(a.x) * fw0 * f.x);
                        s0.y += static_cast<float>(static_cast<double>(a.y) * fw0 * f.y);
                        s1.x += static_cast<float>(static_cast<double>(c.x) * fw1 * f.x);
                        s1.y += static_cast<float>(static_cast<double>(c.y) * fw1 * f.y);
                        acc[bx][n][0] = f32x2_pack(s0.x, s0.y);
                        acc[bx][n][1] = f32x2_pack(s1.x, s1.y);
                    } else {
                        acc[bx][n][0] = f32x2_fma(d01, f32x2_mul(W0, F[n]), acc[bx][n][0]);
                        acc[bx][n][1] = f32x2_fma(d23, f32x2_mul(W1, F[n]), acc[bx][n][1]);
                    }
                }
            }
        }
    }
}

// A full K step (all 8 blocks inside this CTA's range) with every shared
// memory load of the step issued before the unpack / MMA chain, the scale
// bytes of 8 blocks read as one 8-byte word per row (needs K % 256 == 0 so
// the words are aligned), and the activation factors of two blocks per
// 16-byte load.
template <int NT, int BOXES>
__device__ __forceinline__ void consume_step_full(uint32_t slot, uint32_t box_stride, uint32_t sc, int nblk, int kb,
                                                  int kblk0, int ncols, uint32_t xs, uint32_t xs_stride, uint32_t fx,
                                                  uint32_t fx_stride, uint64_t (&acc)[BOXES][NT][2], int lane) {
    const int g = lane >> 2;
    const int tig = lane & 3;
    const int mi = lane >> 3;
    const int row = ((mi & 1) << 3) | (lane & 7);
    const int bsel = mi >> 1;
    uint32_t r[BOXES][4][4];
#pragma unroll
    for (int bx = 0; bx < BOXES; ++bx)
#pragma unroll
        for (int jp = 0; jp < 4; ++jp)
            ldmatrix_x4(slot + bx * box_stride + row * 128 + (((2 * jp + bsel) ^ (row & 7)) << 4), r[bx][jp][0],
                        r[bx][jp][1], r[bx][jp][2], r[bx][jp][3]);
    uint2 s0[BOXES], s1[BOXES];
#pragma unroll
    for (int bx = 0; bx < BOXES; ++bx) {
        const uint32_t scb = sc + bx * 16 * nblk + kb * 8;
        s0[bx] = lds64(scb + g * nblk);
        s1[bx] = lds64(scb + (g + 8) * nblk);
    }
    const int bl0 = kb * 8 - kblk0;
    // Per-lane bases of this step; the 8 blocks are immediate offsets.
    // A lane whose token column does not exist (every unit has at least one)
    // reads the last real column instead: that column of the MMA output only
    // meets zero factors, so it adds nothing, and the load needs no branch.
    uint32_t xb[NT], fb[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        xb[n] = xs + min(g + 8 * n, ncols - 1) * xs_stride + bl0 * 64 + tig * 16;
        fb[n] = fx + (tig + 4 * n) * fx_stride + bl0 * 8;
    }
    uint64_t Fe[NT], Fo[NT];
#pragma unroll
    for (int blk = 0; blk < 8; ++blk) {
        uint4 xv[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            xv[n] = lds128(xb[n] + blk * 64);
            if ((blk & 1) == 0) lds128_pairs(fb[n] + blk * 8, Fe[n], Fo[n]);
        }
        const int jp = blk >> 1, h = blk & 1;
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx) {
            // Byte (blk & 3) of both rows' scale words -> bytes 0 and 1.
            const uint32_t w0 = blk < 4 ? s0[bx].x : s0[bx].y;
            const uint32_t w1 = blk < 4 ? s1[bx].x : s1[bx].y;
            const uint32_t fw = e8m0x2_to_bf16x2(prmt(w0, w1, (blk & 3) | ((4 + (blk & 3)) << 4)));
            const float fw0 = __uint_as_float(fw << 16), fw1 = __uint_as_float(fw & 0xffff0000u);
            const uint64_t W0 = f32x2_pack(fw0, fw0), W1 = f32x2_pack(fw1, fw1);
            uint32_t ga[4], gb[4];
            e2m1x8_to_f16x8(r[bx][jp][2 * h], ga[0], ga[1], ga[2], ga[3]);
            e2m1x8_to_f16x8(r[bx][jp][2 * h + 1], gb[0], gb[1], gb[2], gb[3]);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const uint64_t F = h ? Fo[n] : Fe[n];
                uint64_t d01, d23;
                mma_f16_k32(d01, d23, ga, gb, xv[n]);
                acc[bx][n][0] = f32x2_fma(d01, f32x2_mul(W0, F), acc[bx][n][0]);
                acc[bx][n][1] = f32x2_fma(d23, f32x2_mul(W1, F), acc[bx][n][1]);
            }
        }
    }
}

// Final per-unit sums handed to a problem's epilogue: [box][column][16 rows].
template <int NT>
// A unit's sum for (box, col, row) is the sum, in order, of nparts partial
// arrays part_stride floats apart, each [box][column][row] with row_stride
// floats per column.
struct Sums {
    const float* f;
    int nparts;
    int part_stride;
    int row_stride;
    __device__ float sum(int box, int col, int r) const {
        const float* q = f + (box * 8 * NT + col) * row_stride + r;
        float s = 0.f;
        for (int j = 0; j < nparts; ++j) s += q[j * part_stride];
        return s;
    }
};

// Where a CTA sits: which units, which part of K.
struct Placement {
    int u0, u1;        // units [u0, u1)
    int kb0, kb1;      // K steps [kb0, kb1) (256 values each)
    int kblk0, kblk1;  // 32-blocks [kblk0, kblk1)
    uint32_t rank, cl;
};

// K in parts: one item of a CTA's work is the K steps [kb0, kb1) of part
// `part` of one unit.
struct Item {
    int u;         // unit
    uint32_t uu;   // unit ordinal within the CTA (scale-slot sequence)
    int part;      // K part
    int kb0, kb1;  // K steps (256 values each)
};

// The CTA's items in streaming order: units in batches of ub; for each part,
// that part of every unit of the batch.
struct ItemSeq {
    int u0, nu;
    int ps, nparts, ub;
    int nkb, nblk;
    __device__ int count() const { return nu * nparts; }
    __device__ int nchunks() const { return ((nu + ub - 1) / ub) * nparts; }  // activation parts staged
    __device__ void part_blocks(int part, int& b0, int& b1) const {
        b0 = part * ps * 8;
        b1 = min(nblk, (part + 1) * ps * 8);
    }
    __device__ Item at(int v) const {
        // Every batch but the last is full, so the batch is v / (ub * nparts).
        const int bi = v / (ub * nparts);
        const int r = v - bi * ub * nparts;
        const int bsize = min(ub, nu - bi * ub);
        Item it;
        it.part = r / bsize;
        it.uu = static_cast<uint32_t>(bi * ub + r - it.part * bsize);
        it.u = u0 + static_cast<int>(it.uu);
        it.kb0 = it.part * ps;
        it.kb1 = min(nkb, it.kb0 + ps);
        return it;
    }
};

// ------------------------------------------------------------------------
// Shared-memory carve-up of one CTA (offsets from the 1024-aligned base).
struct Smem {
    uint32_t base;
    uint8_t* gbase;
    SmemLayout L;
    Bars bars;
    WaitCtx wait;
    volatile int* wide;  // see StageDst::wide
};

template <class P>
__device__ void producer_role(const typename P::Params& p, const Smem& S, const Placement& pl,
                              const CUtensorMap* tmap, int lane) {
    // One lane issues everything: per unit one scale copy, per stage (L.steps
    // K steps of BOXES boxes) one expect_tx and the stage's TMA loads. A
    // stage carries 8-16 KB, so the per-copy barrier traffic stays small.
    if (lane != 0) return;
    constexpr int BOXES = P::BOXES;
    const SmemLayout& L = S.L;
    const Bars& bars = S.bars;
    const uint32_t spb = L.steps;
    const uint32_t stage_bytes = spb * BOXES * kBoxBytes;
    const uint32_t scale_bytes = 16u * static_cast<uint32_t>(p.nblk);
    const int nkbc = pl.kb1 - pl.kb0;
    if (nkbc <= 0) return;  // a cluster rank with no part of K: nothing to stream
    const uint64_t policy = l2_evict_first_policy();
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
    bool ok = true;
    uint32_t staged = 0, sissued = 0;
    for (int u = pl.u0; u < pl.u1 && ok; ++u) {
        const uint32_t uu = u - pl.u0;
        const uint32_t ss = uu % L.nss;
        if (!mbar_wait(bars.sempty(ss), ((uu / L.nss) & 1) ^ 1, S.wait)) {
            ok = false;
            break;
        }
        sts_u32_volatile(bars.scale_tag(ss), uu);  // the slot now belongs to unit uu
        // Scale rows of the unit: a bulk copy of the 16-byte-aligned part, and
        // (only for a tail row group) the last few bytes stored by this lane.
        const uint32_t bytes = static_cast<uint32_t>(P::unit_rows(p, u)) * static_cast<uint32_t>(p.nblk);
        const uint32_t bulk = bytes & ~15u;
        const uint32_t dst = S.base + L.sc + ss * L.ss_bytes;
        uint8_t* dst_g = S.gbase + L.sc + ss * L.ss_bytes;
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx) {
            const uint8_t* src = P::scale_src(p, u, bx);
            for (uint32_t b = bulk; b < bytes; ++b) dst_g[bx * scale_bytes + b] = src[b];
        }
        mbar_arrive_expect_tx(bars.sfull(ss), bulk * BOXES);
        if (bulk) {
#pragma unroll
            for (int bx = 0; bx < BOXES; ++bx)
                bulk_load(dst + bx * scale_bytes, P::scale_src(p, u, bx), bulk, bars.sfull(ss), policy);
        }
        ++sissued;
        int rows[BOXES];
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx) rows[bx] = P::box_row(p, u, bx);
        for (int st = 0; st < nkbc; st += static_cast<int>(spb)) {
            const uint32_t slot = staged % L.nslot;
            if (!mbar_wait(bars.empty(slot), ((staged / L.nslot) & 1) ^ 1, S.wait)) {
                ok = false;
                break;
            }
            // The slot now belongs to stage `staged`: its previous stage has
            // been consumed, so a consumer that sees this tag can wait on the
            // slot's full barrier without mistaking an older phase for it.
            sts_u32_volatile(bars.ring_tag(slot), staged);
            if (withhold_stage(staged)) {  // test-only builds
                ++staged;
                continue;
            }
            mbar_arrive_expect_tx(bars.full(slot), stage_bytes);
            const uint32_t sbase = S.base + L.ring + slot * stage_bytes;
            if (p.tma3d >= kCopyMerged3d) {
                // One copy for every box of the stage: [step][box][16 rows][128 B].
                issue_merged_stage(p.tma3d, sbase, tmap, rows[0], pl.kb0 + st, bars.full(slot), policy);
            } else if (p.tma3d) {
                // Stage layout [box][step][16 rows][128 B], 128-byte swizzle: one
                // copy per box of 16 rows x spb 128-byte segments of K.
#pragma unroll
                for (int bx = 0; bx < BOXES; ++bx)
                    tma_load_3d(sbase + bx * spb * kBoxBytes, tmap, 0, rows[bx], pl.kb0 + st, bars.full(slot),
                                policy);
            } else {
                for (uint32_t j = 0; j < spb; ++j) {
                    const int kb = pl.kb0 + st + static_cast<int>(j);
#pragma unroll
                    for (int bx = 0; bx < BOXES; ++bx)
                        tma_load_2d(sbase + (bx * spb + j) * kBoxBytes, tmap, kb * 128, rows[bx], bars.full(slot),
                                    policy);
                }
            }
            ++staged;
        }
    }
    if (!ok) {
        // Let every copy still in flight land (bounded) before the CTA exits.
        // These waits ignore the abort flag: copies complete on their own.
        int never = 0;
        const WaitCtx own{p.status, &never};
        const uint32_t first = staged > L.nslot ? staged - L.nslot : 0;
        for (uint32_t j = first; j < staged; ++j) mbar_wait(bars.full(j % L.nslot), (j / L.nslot) & 1, own);
        const uint32_t sfirst = sissued > L.nss ? sissued - L.nss : 0;
        for (uint32_t j = sfirst; j < sissued; ++j) mbar_wait(bars.sfull(j % L.nss), (j / L.nss) & 1, own);
    }
}

template <class P>
__device__ void producer_parts(const typename P::Params& p, const Smem& S, const Placement& pl, const ItemSeq& seq,
                               const CUtensorMap* tmap, int lane) {
    // producer_role over the items of K in parts: a unit's scales (all of
    // K) are copied with its first part and serve every part; the stages of
    // each item follow in streaming order.
    if (lane != 0) return;
    constexpr int BOXES = P::BOXES;
    const SmemLayout& L = S.L;
    const Bars& bars = S.bars;
    const uint32_t spb = L.steps;
    const uint32_t stage_bytes = spb * BOXES * kBoxBytes;
    const uint32_t scale_bytes = 16u * static_cast<uint32_t>(p.nblk);
    if (pl.kb1 - pl.kb0 <= 0) return;  // a cluster rank with no part of K: nothing to stream
    const uint64_t policy = l2_evict_first_policy();
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
    bool ok = true;
    uint32_t staged = 0, sissued = 0;
    uint32_t slot = 0, rph = 0;  // ring slot of stage `staged` and its round parity
    uint32_t ss = 0, sph = 0;    // scale slot of the next unit's first part and its round parity
    const int ni = seq.count();
    for (int v = 0; v < ni && ok; ++v) {
        const Item it = seq.at(v);
        const int u = it.u;
        const uint32_t uu = it.uu;
        if (it.part == 0) {
            if (!mbar_wait(bars.sempty(ss), sph ^ 1, S.wait)) {
                ok = false;
                break;
            }
            sts_u32_volatile(bars.scale_tag(ss), uu);  // the slot now belongs to unit uu
            // Scale rows of the unit: a bulk copy of the 16-byte-aligned part, and
            // (only for a tail row group) the last few bytes stored by this lane.
            const uint32_t bytes = static_cast<uint32_t>(P::unit_rows(p, u)) * static_cast<uint32_t>(p.nblk);
            const uint32_t bulk = bytes & ~15u;
            const uint32_t dst = S.base + L.sc + ss * L.ss_bytes;
            uint8_t* dst_g = S.gbase + L.sc + ss * L.ss_bytes;
#pragma unroll
            for (int bx = 0; bx < BOXES; ++bx) {
                const uint8_t* src = P::scale_src(p, u, bx);
                for (uint32_t b = bulk; b < bytes; ++b) dst_g[bx * scale_bytes + b] = src[b];
            }
            mbar_arrive_expect_tx(bars.sfull(ss), bulk * BOXES);
            if (bulk) {
#pragma unroll
                for (int bx = 0; bx < BOXES; ++bx)
                    bulk_load(dst + bx * scale_bytes, P::scale_src(p, u, bx), bulk, bars.sfull(ss), policy);
            }
            ++sissued;
            ring_next(ss, sph, L.nss);
        }
        int rows[BOXES];
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx) rows[bx] = P::box_row(p, u, bx);
        for (int kb = it.kb0; kb < it.kb1; kb += static_cast<int>(spb)) {
            if (!mbar_wait(bars.empty(slot), rph ^ 1, S.wait)) {
                ok = false;
                break;
            }
            // The slot now belongs to stage `staged`: its previous stage has
            // been consumed, so a consumer that sees this tag can wait on the
            // slot's full barrier without mistaking an older phase for it.
            sts_u32_volatile(bars.ring_tag(slot), staged);
            mbar_arrive_expect_tx(bars.full(slot), stage_bytes);
            const uint32_t sbase = S.base + L.ring + slot * stage_bytes;
            if (p.tma3d >= kCopyMerged3d) {
                issue_merged_stage(p.tma3d, sbase, tmap, rows[0], kb, bars.full(slot), policy);
            } else if (p.tma3d) {
                // Stage layout [box][step][16 rows][128 B]: one copy per box.
#pragma unroll
                for (int bx = 0; bx < BOXES; ++bx)
                    tma_load_3d(sbase + bx * spb * kBoxBytes, tmap, 0, rows[bx], kb, bars.full(slot), policy);
            } else {
                for (uint32_t j = 0; j < spb; ++j) {
#pragma unroll
                    for (int bx = 0; bx < BOXES; ++bx)
                        tma_load_2d(sbase + (bx * spb + j) * kBoxBytes, tmap, (kb + static_cast<int>(j)) * 128,
                                    rows[bx], bars.full(slot), policy);
                }
            }
            ++staged;
            ring_next(slot, rph, L.nslot);
        }
    }
    if (!ok) {
        // Let every copy still in flight land (bounded) before the CTA exits.
        // These waits ignore the abort flag: copies complete on their own.
        int never = 0;
        const WaitCtx own{p.status, &never};
        const uint32_t first = staged > L.nslot ? staged - L.nslot : 0;
        for (uint32_t j = first; j < staged; ++j) mbar_wait(bars.full(j % L.nslot), (j / L.nslot) & 1, own);
        const uint32_t sfirst = sissued > L.nss ? sissued - L.nss : 0;
        for (uint32_t j = sfirst; j < sissued; ++j) mbar_wait(bars.sfull(j % L.nss), (j / L.nss) & 1, own);
    }
}

// Consumer warps that own chunks of each unit on cluster rank q (the same
// split of K steps the placement uses).
__device__ __forceinline__ int rank_owners(int nkb, int cl, int q, int group, int ncw) {
    const int nkb_c = (nkb + cl - 1) / cl;
    const int k0 = min(nkb, q * nkb_c);
    const int k1 = min(nkb, k0 + nkb_c);
    return min((k1 - k0) / group, ncw);
}

template <class P>
__device__ void consumer_role(const typename P::Params& p, const Smem& S, const Placement& pl, int warp, int lane) {
    constexpr int NT = P::NT;
    constexpr int BOXES = P::BOXES;
    constexpr int kRedWarpFloats = BOXES * 8 * NT * kRedStride;
    const SmemLayout& L = S.L;
    const Bars& bars = S.bars;
    const uint32_t spb = L.steps;
    const uint32_t G = L.group;
    const uint32_t stage_bytes = spb * BOXES * kBoxBytes;
    uint8_t* xs = S.gbase + L.xs;
    float* fx = reinterpret_cast<float*>(S.gbase + L.fx);
    float* redw = reinterpret_cast<float*>(S.gbase + L.red);
    const uint32_t xs_s = S.base + L.xs, fx_s = S.base + L.fx, scb = S.base + L.sc;
    const int nkbc = pl.kb1 - pl.kb0;
    const bool fast_steps = (p.nblk & 7) == 0;  // 8-byte aligned scale words
    int cur_chunk = -1;
    int ncols = 0;
    uint32_t xphase = 0;
    // The CTA's K steps, unit after unit, are cut into chunks of G steps
    // (G divides the stage size spb, which divides a unit's steps, so a chunk
    // never straddles two stages or two units). This warp takes chunks c =
    // warp, warp + NCW, ...; chunk c is chunk `within` of stage c / cps,
    // which sits in ring slot stage % nslot.
    const uint32_t cps = spb / G;
    const uint32_t cpu = static_cast<uint32_t>(nkbc) / G;
    // Partial slots of a unit: rank q's owners use [base_q, base_q + owners_q)
    // of the buffer on rank 0; `total` counts every rank's owners.
    const int ranks = static_cast<int>(pl.cl);
    uint32_t rbase = 0, total = 0;
    for (int q = 0; q < ranks; ++q) {
        const uint32_t o = static_cast<uint32_t>(rank_owners(p.nkb, ranks, q, static_cast<int>(G), P::NCW));
        if (q < static_cast<int>(pl.rank)) rbase += o;
        total += o;
    }
    const bool lone = pl.cl == 1;
    const uint32_t red0 = lone ? S.base + L.red : map_to_rank(S.base + L.red, 0);  // rank 0's buffers
    const uint32_t count0 = lone ? 0u : map_to_rank(bars.red_count(0), 0);
    const uint32_t ring = S.base + L.ring;
    // Stage layout [box][step] (per-box copies) or [step][box] (one copy).
    const bool merged = p.tma3d >= kCopyMerged3d;
    const uint32_t box_stride = merged ? kBoxBytes : spb * kBoxBytes;
    const uint32_t step_bytes = merged ? BOXES * kBoxBytes : kBoxBytes;
    const uint32_t adv_stage = P::NCW / cps, adv_within = P::NCW - (P::NCW / cps) * cps;
    uint32_t c = warp;
    uint32_t within = c % cps;
    uint32_t stage = c / cps;
    uint32_t slot = stage % L.nslot;
    uint32_t phase = (stage / L.nslot) & 1u;
    uint32_t ss = 0, sph = 0;  // scale slot of unit uu and its round parity
    uint32_t rb = 0, rph = 0;  // reduction buffer of unit uu (uu % nrb)
    for (int u = pl.u0; u < pl.u1; ++u, ring_next(ss, sph, L.nss), ring_next(rb, rph, L.nrb)) {
        const uint32_t uu = u - pl.u0;
        const int chunk = P::chunk_of(p, u);
        if (cur_chunk < 0) pdl_wait_previous();  // activations may come from the previous kernel
        if (chunk != cur_chunk) {
            if constexpr (HasInputGate<P>::value) {
                if (!__all_sync(0xffffffffu, P::wait_inputs(p, S.wait))) return;
            }
            // Everyone is done with the previous columns before they change,
            // and the new ones are complete before anyone reads them. The
            // barriers are mbarriers so a wait can give up instead of hang.
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.xbar(0));
            if (!warp_wait(bars.xbar(0), xphase & 1, S.wait)) return;
            const StageDst dst{xs, reinterpret_cast<uint8_t*>(fx), L.xs_stride, L.fx_stride, S.wide};
            if constexpr (P::kBulkStage) {
                if (!stage_bulk<P>(p, chunk, pl.kblk0, pl.kblk1, dst, xs_s, bars.xbar(2), xphase & 1, S.wait,
                                   warp * 32 + lane, Roles<P>::kConsumerThreads))
                    return;
            } else {
                P::stage(p, chunk, pl.kblk0, pl.kblk1, dst, warp * 32 + lane, Roles<P>::kConsumerThreads);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.xbar(1));
            if (!warp_wait(bars.xbar(1), xphase & 1, S.wait)) return;
            ++xphase;
            cur_chunk = chunk;
            ncols = P::ncols(p, chunk);
        }
        const uint32_t cb = uu * cpu;  // first chunk of this unit
        // A warp owns chunks of this unit iff its next chunk lies inside it;
        // its partial goes to slot c - cb (< NCW, since its previous chunk
        // lies before the unit).
        // Only owners take part in the unit: they wait for its scales, hand
        // in their partial and release the scale slot.
        if (c >= cb + cpu) continue;
        const uint32_t jred = c - cb;
        uint64_t acc[BOXES][NT][2];
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx)
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[bx][n][0] = acc[bx][n][1] = 0ull;  // +0.0f pairs
        {
            // This warp may be several units ahead of the scale ring: the tag
            // says the slot holds this unit's scales (or is being filled).
            if (!__all_sync(0xffffffffu, wait_shared_value(bars.scale_tag(ss), uu, S.wait))) return;
            if (!warp_wait(bars.sfull(ss), sph, S.wait)) return;
            const uint32_t sc = scb + ss * L.ss_bytes;
            for (; c < cb + cpu; c += P::NCW) {
                // A warp may run several stages ahead of the ring: first wait
                // until the producer has claimed the slot for this stage, so
                // the parity wait below refers to this stage's phase.
                if (!__all_sync(0xffffffffu, wait_shared_value(bars.ring_tag(slot), stage, S.wait))) return;
                if (!warp_wait(bars.full(slot), phase, S.wait)) return;
                uint32_t step_smem = ring + slot * stage_bytes + within * G * step_bytes;
                int kb = pl.kb0 + static_cast<int>((c - cb) * G);
                const bool wide = *S.wide != 0;  // stable once this chunk's activations are staged
                for (uint32_t st = 0; st < G; ++st, ++kb, step_smem += step_bytes) {
                    if (wide)
                        consume_step<NT, BOXES, true>(step_smem, box_stride, sc, p.nblk, kb, pl.kblk0, pl.kblk1,
                                                      ncols, xs_s, L.xs_stride, fx_s, L.fx_stride, acc, lane);
                    else if (fast_steps && kb * 8 + 8 <= pl.kblk1)
                        consume_step_full<NT, BOXES>(step_smem, box_stride, sc, p.nblk, kb, pl.kblk0, ncols, xs_s,
                                                     L.xs_stride, fx_s, L.fx_stride, acc, lane);
                    else
                        consume_step<NT, BOXES>(step_smem, box_stride, sc, p.nblk, kb, pl.kblk0, pl.kblk1, ncols,
                                                xs_s, L.xs_stride, fx_s, L.fx_stride, acc, lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.empty(slot));
                // Next chunk of this warp: c + NCW, i.e. (stage, within)
                // advanced without a division.
                within += adv_within;
                uint32_t ds = adv_stage;
                if (within >= cps) {
                    within -= cps;
                    ++ds;
                }
                stage += ds;
                slot += ds;
                while (slot >= L.nslot) {
                    slot -= L.nslot;
                    phase ^= 1u;
                }
            }
        }
        // Reduction buffer uu % nrb (on rank 0) is free once unit uu - nrb is
        // finished; its finisher tags the buffer on every rank.
        if (!__all_sync(0xffffffffu, wait_shared_value(bars.red_tag(rb), uu - L.nrb, S.wait))) return;
        if (lone)
            __threadfence_block();
        else
            fence_acq_rel_cluster();
        {
            const uint32_t slot_f = (rb * L.nred_all + rbase + jred) * kRedWarpFloats;
            const int g = lane >> 2, tig = lane & 3;
#pragma unroll
            for (int bx = 0; bx < BOXES; ++bx)
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint32_t rb_f = slot_f + (bx * 8 * NT + 8 * n + 2 * tig) * kRedStride;
                    const float2 a01 = f32x2_unpack(acc[bx][n][0]), a23 = f32x2_unpack(acc[bx][n][1]);
                    if (lone) {
                        float* Rb = redw + rb_f;
                        Rb[g] = a01.x;
                        Rb[kRedStride + g] = a01.y;
                        Rb[g + 8] = a23.x;
                        Rb[kRedStride + g + 8] = a23.y;
                    } else {
                        st_cluster_f32(red0 + 4 * (rb_f + g), a01.x);
                        st_cluster_f32(red0 + 4 * (rb_f + kRedStride + g), a01.y);
                        st_cluster_f32(red0 + 4 * (rb_f + g + 8), a23.x);
                        st_cluster_f32(red0 + 4 * (rb_f + kRedStride + g + 8), a23.y);
                    }
                }
        }
        __syncwarp();
        // Count the hand-in. Lone CTA: the owner that completes the count
        // finishes the unit. Cluster: rank 0's first owner of the unit waits
        // for every rank's partials and finishes it.
        uint32_t prev = 0;
        if (lane == 0) {
            if (lone) {
                __threadfence_block();
                prev = atom_add_shared(bars.red_count(rb), 1u);
            } else {
                fence_acq_rel_cluster();
                prev = atom_add_cluster(count0 + 4 * rb, 1u);
            }
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        bool finish = lone ? prev + 1 == total : (pl.rank == 0 && jred == 0);
        if (finish && !lone) {
            if (!__all_sync(0xffffffffu, wait_shared_value(bars.red_count(rb), total, S.wait))) return;
        }
        if (finish) {
            if (lone)
                __threadfence_block();
            else
                fence_acq_rel_cluster();
            // Sum of the slots in order: rank 0's owners in K order, then
            // rank 1's, ... (deterministic).
            P::epilogue(p, u,
                        Sums<NT>{redw + rb * L.nred_all * kRedWarpFloats, static_cast<int>(total), kRedWarpFloats,
                                 kRedStride},
                        lane);
            __syncwarp();
            if (lane == 0) sts_u32_volatile(bars.red_count(rb), 0);
            if (lone) {
                if (lane == 0) {
                    __threadfence_block();
                    sts_u32_volatile(bars.red_tag(rb), uu);
                }
            } else {
                fence_acq_rel_cluster();
                if (lane < ranks) st_cluster_u32(map_to_rank(bars.red_tag(rb), static_cast<uint32_t>(lane)), uu);
            }
        }
        if (lane == 0) mbar_arrive(bars.sempty(ss));
    }
}

// K in parts (lone CTA): the units of a batch belong to one warp each (warp
// j takes unit j of every batch; ub <= NCW), so a unit's accumulators stay
// in that warp's registers across all parts and its epilogue runs once.
// Every consumer warp, owner or not, takes part in staging each part's
// activations: the part's buffer (q & 1 for chunk q = batch * nparts + part)
// was filled by a copy that the last warp to leave chunk q - 2 issued (the
// first thread issues chunks 0 and 1); each warp converts its share, and all
// shares are done before any warp reads the buffer.
template <class P>
__device__ void consumer_parts(const typename P::Params& p, const Smem& S, const ItemSeq& seq, int warp, int lane) {
    constexpr int NT = P::NT;
    constexpr int BOXES = P::BOXES;
    constexpr int kRedWarpFloats = BOXES * 8 * NT * kRedStride;
    const SmemLayout& L = S.L;
    const Bars& bars = S.bars;
    const uint32_t spb = L.steps;
    const uint32_t stage_bytes = spb * BOXES * kBoxBytes;
    const bool merged = p.tma3d >= kCopyMerged3d;  // stage layout [step][box] instead of [box][step]
    const uint32_t box_stride = merged ? kBoxBytes : spb * kBoxBytes;
    const uint32_t step_bytes = merged ? BOXES * kBoxBytes : kBoxBytes;
    const uint32_t spi = L.part_steps / spb;  // stages per item
    uint8_t* xs = S.gbase + L.xs;
    uint8_t* fx = S.gbase + L.fx;
    float* red = reinterpret_cast<float*>(S.gbase + L.red) + warp * kRedWarpFloats;  // this warp's slot
    const uint32_t xs_s = S.base + L.xs, fx_s = S.base + L.fx, scb = S.base + L.sc, ring = S.base + L.ring;
    const int tid = warp * 32 + lane;
    const bool fast_steps = (p.nblk & 7) == 0;  // 8-byte aligned scale words
    const int ncols = P::ncols(p, 0);
    const int nq = seq.nchunks();
    pdl_wait_previous();  // activations may come from the previous kernel
    if (tid == 0) {
        for (int q0 = 0; q0 < 2 && q0 < nq; ++q0) {
            int b0, b1;
            seq.part_blocks(q0 % seq.nparts, b0, b1);
            sts_u32_volatile(bars.xissued(q0), 1u);
            issue_column_copies<P>(p, 0, b0, b1, xs_s + q0 * L.xs_buf, L.xs_stride, bars.xbar(q0));
        }
    }
    int q = 0;
    const int nbatch = (seq.nu + seq.ub - 1) / seq.ub;
    for (int bi = 0; bi < nbatch; ++bi) {
        const int bsize = min(seq.ub, seq.nu - bi * seq.ub);
        const bool own = warp < bsize;
        const uint32_t uu = static_cast<uint32_t>(bi * seq.ub + warp);
        const uint32_t ss = uu % L.nss;
        uint64_t acc[BOXES][NT][2];
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx)
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[bx][n][0] = acc[bx][n][1] = 0ull;  // +0.0f pairs
        for (int part = 0; part < seq.nparts; ++part, ++q) {
            if (q > 0) {
                // This warp has left chunk q - 1: the last warp out reloads
                // that buffer with chunk q + 1.
                __syncwarp();
                if (lane == 0) {
                    const uint32_t b = static_cast<uint32_t>(q - 1) & 1u;
                    __threadfence_block();  // this warp's reads of the buffer come first
                    if (atom_add_shared(bars.xdone(b), 1u) == static_cast<uint32_t>(P::NCW - 1)) {
                        sts_u32_volatile(bars.xdone(b), 0u);
                        if (q + 1 < nq) {
                            __threadfence_block();
                            int b0, b1;
                            seq.part_blocks((q + 1) % seq.nparts, b0, b1);
                            sts_u32_volatile(bars.xissued(b), lds_u32_volatile(bars.xissued(b)) + 1u);
                            issue_column_copies<P>(p, 0, b0, b1, xs_s + b * L.xs_buf, L.xs_stride, bars.xbar(b));
                        }
                    }
                }
            }
            int kblk0, kblk1;
            seq.part_blocks(part, kblk0, kblk1);
            const uint32_t b = static_cast<uint32_t>(q) & 1u;
            const uint32_t par = (static_cast<uint32_t>(q) >> 1) & 1u;
            if (!warp_wait(bars.xbar(b), par, S.wait)) return;
            const StageDst dst{xs + b * L.xs_buf, fx + b * L.fx_buf, L.xs_stride, L.fx_stride, S.wide};
            convert_columns<8 * NT>(P::stage_cols(p, 0), kblk1 - kblk0, dst, xs_s + b * L.xs_buf, tid,
                                    Roles<P>::kConsumerThreads);
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.xbar(2 + b));
            if (!warp_wait(bars.xbar(2 + b), par, S.wait)) return;
            if (!own) continue;
            if (part == 0) {
                // The unit's scales (all of K) arrive with its first part.
                if (!__all_sync(0xffffffffu, wait_shared_value(bars.scale_tag(ss), uu, S.wait))) return;
                if (!warp_wait(bars.sfull(ss), (uu / L.nss) & 1, S.wait)) return;
            }
            const uint32_t sc = scb + ss * L.ss_bytes;
            const uint32_t xcur = xs_s + b * L.xs_buf, fcur = fx_s + b * L.fx_buf;
            // The producer streams item (batch, part, unit) as item number
            // v = (batch * nparts + part) * ub + unit of a full batch (the
            // last batch has bsize units), spi stages each.
            const uint32_t v = static_cast<uint32_t>(bi * seq.ub * seq.nparts + part * bsize + warp);
            uint32_t stage = v * spi;
            int kb = part * seq.ps;
            for (uint32_t s = 0; s < spi; ++s, ++stage) {
                const uint32_t slot = stage % L.nslot;
                const uint32_t phase = (stage / L.nslot) & 1u;
                // The tag says the producer has claimed the slot for this
                // stage, so the parity wait refers to this stage's phase.
                if (!__all_sync(0xffffffffu, wait_shared_value(bars.ring_tag(slot), stage, S.wait))) return;
                if (!warp_wait(bars.full(slot), phase, S.wait)) return;
                uint32_t step_smem = ring + slot * stage_bytes;
                const bool wide = *S.wide != 0;  // stable once this part's activations are staged
                for (uint32_t st = 0; st < spb; ++st, ++kb, step_smem += step_bytes) {
                    if (wide)
                        consume_step<NT, BOXES, true>(step_smem, box_stride, sc, p.nblk, kb, kblk0, kblk1, ncols,
                                                      xcur, L.xs_stride, fcur, L.fx_stride, acc, lane);
                    else if (fast_steps && kb * 8 + 8 <= kblk1)
                        consume_step_full<NT, BOXES>(step_smem, box_stride, sc, p.nblk, kb, kblk0, ncols, xcur,
                                                     L.xs_stride, fcur, L.fx_stride, acc, lane);
                    else
                        consume_step<NT, BOXES>(step_smem, box_stride, sc, p.nblk, kb, kblk0, kblk1, ncols, xcur,
                                                L.xs_stride, fcur, L.fx_stride, acc, lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.empty(slot));
            }
        }
        if (own) {
            // All of K is in the registers: through this warp's own slot to
            // the problem's epilogue.
            const int g = lane >> 2, tig = lane & 3;
#pragma unroll
            for (int bx = 0; bx < BOXES; ++bx)
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    float* Rb = red + (bx * 8 * NT + 8 * n + 2 * tig) * kRedStride;
                    const float2 a01 = f32x2_unpack(acc[bx][n][0]), a23 = f32x2_unpack(acc[bx][n][1]);
                    Rb[g] = a01.x;
                    Rb[kRedStride + g] = a01.y;
                    Rb[g + 8] = a23.x;
                    Rb[kRedStride + g + 8] = a23.y;
                }
            __syncwarp();
            P::epilogue(p, seq.u0 + static_cast<int>(uu), Sums<NT>{red, 1, kRedWarpFloats, kRedStride}, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.sempty(ss));
        }
    }
}

// ------------------------------------------------------------------------
// The kernel. P (the problem) supplies:
//   static constexpr int NT, BOXES;
//   struct Params { ...; unsigned* status; int nblk; int nkb; int xcols; int cl; int tma3d; SmemLayout layout; };
//     xcols = staged columns (the layout's column count)
//     tma3d = the tensor map is the 3D view (128 B, rows, K/256 segments) and one
//     copy fetches a whole stage of a box; else it is the 2D view (K/2 B, rows).
//     (stage() writes through StageDst and zeroes the factors of unused columns);
//     cl = CTAs per cluster splitting K; layout.part_steps > 0 walks K in parts
//     (lone CTAs of bulk-staged problems only).
//   __device__ static int  num_units(const Params&);
//   __device__ static int  chunk_of(const Params&, int u);
//   __device__ static int  box_row(const Params&, int u, int box);      // TMA row coordinate
//   __device__ static const uint8_t* scale_src(const Params&, int u, int box);
//   __device__ static int  unit_rows(const Params&, int u);            // valid rows (<= 16)
//   __device__ static int  ncols(const Params&, int chunk);            // staged columns
//   __device__ static void stage(const Params&, int chunk, int kblk0, int kblk1, const StageDst&,
//                                int tid, int nthreads);
//   __device__ static void epilogue(const Params&, int u, const Sums<NT>&, int lane);
//   optional: static constexpr bool kInputGate = true; and
//   __device__ static bool wait_inputs(const Params&, const WaitCtx&) -- called by
//   every consumer warp before it stages a chunk's activations (a problem whose
//   activations another CTA of the same grid produces waits for them there;
//   false = the wait gave up).
// stream_body is the whole CTA program; a kernel may run it more than once
// (one problem after another) on the same shared memory.
template <class P, bool kParts>
__device__ __forceinline__ void stream_body(const CUtensorMap& tmap, const typename P::Params& p,
                                            uint8_t* smem_raw) {
    const uint32_t raw = smem_addr(smem_raw);
    Smem S;
    S.base = (raw + 1023u) & ~1023u;
    S.gbase = smem_raw + (S.base - raw);
    S.L = p.layout;
    S.bars = Bars{S.base + S.L.bars, S.L.nslot, S.L.nss, S.L.nrb, S.base + S.L.tags};
    S.wait = WaitCtx{p.status, reinterpret_cast<volatile int*>(S.gbase + (S.bars.abort_flag() - S.base))};
    S.wide = reinterpret_cast<volatile int*>(S.gbase + (S.bars.abort_flag() + 4 - S.base));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The next kernel on the stream may be scheduled now: it only streams
    // weights until it has waited for this kernel (pdl_wait_previous).
    pdl_launch_dependents();

    Placement pl;
    pl.cl = p.cl > 1 ? static_cast<uint32_t>(p.cl) : 1u;
    pl.rank = pl.cl > 1 ? cluster_ctarank() : 0u;
    const int ngroups = pl.cl > 1 ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
    const int group = pl.cl > 1 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int nkb_c = (p.nkb + static_cast<int>(pl.cl) - 1) / static_cast<int>(pl.cl);
    pl.kb0 = min(p.nkb, static_cast<int>(pl.rank) * nkb_c);
    pl.kb1 = min(p.nkb, pl.kb0 + nkb_c);
    pl.kblk0 = pl.kb0 * 8;
    pl.kblk1 = min(p.nblk, pl.kb1 * 8);

    if (warp == 0) {
        // Warp 0 initialises the barriers and tags, one lane per ring / scale
        // slot; each lane fences its own inits.
        const Bars& bars = S.bars;
        // Warps that own chunks of a unit: the arrivals its reduction buffer
        // and scale slot wait for (at least 1 so the count is valid; a rank
        // with no K steps has no owners and never waits on them). K in parts:
        // one owner per unit.
        const int cpu = (pl.kb1 - pl.kb0) / static_cast<int>(S.L.group);
        const uint32_t nown = kParts ? 1u : static_cast<uint32_t>(max(1, min(cpu, P::NCW)));
        for (uint32_t s = lane; s < S.L.nslot; s += 32) {
            mbar_init(bars.full(s), 1);
            mbar_init(bars.empty(s), S.L.steps / S.L.group);  // one arrival per consumer chunk of the stage
            sts_u32_volatile(bars.ring_tag(s), 0xffffffffu);
        }
        for (uint32_t s = lane; s < S.L.nss; s += 32) {
            mbar_init(bars.sfull(s), 1);
            mbar_init(bars.sempty(s), nown);
            sts_u32_volatile(bars.scale_tag(s), 0xffffffffu);
        }
        if (lane < S.L.nrb) {
            sts_u32_volatile(bars.red_tag(lane), lane - S.L.nrb);  // "unit lane - nrb" released it
            sts_u32_volatile(bars.red_count(lane), 0);
        }
        if constexpr (kParts) {
            if (lane < 2) {
                mbar_init(bars.xbar(lane), 1);           // copy of buffer `lane` landed
                mbar_init(bars.xbar(2 + lane), P::NCW);  // buffer `lane` converted
                sts_u32_volatile(bars.xdone(lane), 0);
                sts_u32_volatile(bars.xissued(lane), 0);
            }
        } else {
            if (lane < 2) mbar_init(bars.xbar(lane), P::NCW);  // staging
            if (lane == 2) mbar_init(bars.xbar(2), 1);
        }
        if (lane == 4) {
            *S.wait.abort = 0;
            *S.wide = 0;
        }
        fence_barrier_init();  // visible to the bulk-copy (async) proxy and to cluster peers
    }
    if (pl.cl > 1)
        cluster_sync_all();
    else
        __syncthreads();

    const int U = P::num_units(p);
    pl.u0 = static_cast<int>((int64_t)U * group / ngroups);
    pl.u1 = static_cast<int>((int64_t)U * (group + 1) / ngroups);

    if constexpr (kParts) {
        // K in parts (lone CTAs of bulk-staged problems; the launcher checks).
        ItemSeq seq;
        seq.u0 = pl.u0;
        seq.nu = pl.u1 - pl.u0;
        seq.ps = static_cast<int>(S.L.part_steps);
        seq.nparts = (p.nkb + seq.ps - 1) / seq.ps;
        seq.ub = static_cast<int>(S.L.ubatch);
        seq.nkb = p.nkb;
        seq.nblk = p.nblk;
        if (warp == Roles<P>::kProducer)
            producer_parts<P>(p, S, pl, seq, &tmap, lane);
        else
            consumer_parts<P>(p, S, seq, warp, lane);
        __syncwarp();  // the producer's idle lanes wait for lane 0
        // After a timeout a buffer's last copy may not have been waited for;
        // let it land (bounded, whatever the abort flag says) before the CTA
        // exits. At most one copy per buffer is outstanding.
        __syncthreads();
        if (threadIdx.x == 0) {
            int never = 0;
            const WaitCtx own{p.status, &never};
            for (uint32_t b = 0; b < 2; ++b) {
                const uint32_t n = lds_u32_volatile(S.bars.xissued(b));
                if (n) mbar_wait(S.bars.xbar(b), (n - 1) & 1, own);
            }
        }
    } else {
        if (warp == Roles<P>::kProducer)
            producer_role<P>(p, S, pl, &tmap, lane);
        else
            consumer_role<P>(p, S, pl, warp, lane);

        // No CTA of a cluster leaves while another may still write to it.
        if (pl.cl > 1) cluster_sync_all();
    }
}

// Between two stream_body runs on the same shared memory, after every
// thread of the CTA has left the first one and passed a __syncthreads:
// returns whether that run gave up (its abort flag), and warp 0 invalidates
// the mbarriers it initialised. The caller synchronises the CTA again before
// the next run initialises its own.
__device__ __forceinline__ bool stream_smem_release(const SmemLayout& L, uint8_t* smem_raw, bool parts) {
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const Bars bars{base + L.bars, L.nslot, L.nss, L.nrb, base + L.tags};
    const bool aborted = *reinterpret_cast<volatile int*>(smem_raw + (bars.abort_flag() - raw)) != 0;
    if (threadIdx.x < 32) {
        for (uint32_t s = threadIdx.x; s < L.nslot; s += 32) {
            mbar_inval(bars.full(s));
            mbar_inval(bars.empty(s));
        }
        for (uint32_t s = threadIdx.x; s < L.nss; s += 32) {
            mbar_inval(bars.sfull(s));
            mbar_inval(bars.sempty(s));
        }
        if (threadIdx.x < (parts ? 4u : 3u)) mbar_inval(bars.xbar(threadIdx.x));
    }
    return aborted;
}

template <class P, bool kParts>
__global__ void __launch_bounds__(Roles<P>::kThreads, 1)
    stream_kernel(const __grid_constant__ CUtensorMap tmap, const typename P::Params p) {
    extern __shared__ uint8_t smem_raw[];
    stream_body<P, kParts>(tmap, p, smem_raw);
}

// Host launcher: one CTA per SM (or clusters of p.cl CTAs), never more
// groups than units.
// kParts = the layout walks K in parts (lone CTAs, p.cl == 1).
template <class Prob, bool kParts = false>
cudaError_t launch_stream_kernel(const CUtensorMap& tmap, const typename Prob::Params& p, int units, int num_sms,
                                 cudaStream_t stream) {
    static_assert(!kParts || Prob::kBulkStage, "K in parts stages its activations by bulk copy");
    if ((p.layout.part_steps != 0) != kParts || (kParts && p.cl > 1)) return cudaErrorInvalidValue;
    static int configured[64] = {0};  // dynamic smem already allowed, per device
    static int clusters_cached[64][9] = {};  // co-resident clusters per device and size
    const int smem = static_cast<int>(p.layout.total) + 1024;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || configured[dev] < smem) {
        cudaError_t e = cudaFuncSetAttribute(stream_kernel<Prob, kParts>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = smem;
    }
    const int cl = p.cl > 1 ? p.cl : 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(Roles<Prob>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    // Programmatic dependent launch: this kernel may start (and stream
    // weights) while the previous kernel of the stream finishes.
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int groups = num_sms;
    if (cl > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cl;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        cfg.gridDim = dim3(cl * (num_sms / cl));
        int nclusters = (dev >= 0 && dev < 64 && cl <= 8) ? clusters_cached[dev][cl] : 0;
        if (nclusters == 0) {
            cudaError_t e = cudaOccupancyMaxActiveClusters(&nclusters, stream_kernel<Prob, kParts>, &cfg);
            if (e != cudaSuccess) return e;
            if (nclusters < 1) return cudaErrorInvalidConfiguration;
            if (dev >= 0 && dev < 64 && cl <= 8) clusters_cached[dev][cl] = nclusters;
        }
        groups = nclusters;
    }
    if (groups > units) groups = units;
    if (groups < 1) groups = 1;
    cfg.gridDim = dim3(groups * cl);
    cudaError_t e = cudaLaunchKernelEx(&cfg, stream_kernel<Prob, kParts>, tmap, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mxfp4
