// Packed-E2M1 tensor-core weight-streaming linear layer for sm_103a, 1 <= T <= 8.
//
// What it computes ("Zyphra Inference Wave 2", sections "Speculative
// decoding" and "Quantization"; AMD "megakernel-intro", section "3.
// Low-Precision Data Types"):
//   y[t][n] = bf16( sum_k x[t][k] * w[n][k] ),  w = e2m1(code) * 2^(s-127)
// reading every weight byte from HBM once, for the handful of tokens of a
// decode / verify step.
//
// The weights go to the tensor cores exactly as stored: one TMA copy per
// stage lands packed codes (two per byte) in shared memory with the 128-byte
// swizzle, and tcgen05.mma kind::mxf4 reads them there with their E8M0
// scales from TMEM, so no instruction ever touches a weight byte. kind::mxf4
// takes E2M1 on both sides, so each bf16 activation is written exactly as a
// sum of eight E2M1 digit pieces under one power of two per (token, 32-value
// block). With E = floor(log2 max|x|) of the block (at least -112):
//   X = rne(|x| * 2^(15-E))        a 16-bit integer, exact whenever |x| is
//                                  within 2^8 of the block maximum (a bf16
//                                  value has 8 significant bits);
//   X = sum_{p<8} D_p * 4^(7-p),   D_p in {0, 1, 2, 3};
//   x = sign * sum_p (D_p / 2) * 2^(E - 2p).
// D_p / 2 is an E2M1 value (code D_p, sign in bit 3), so piece p is an E2M1
// row with block scale 2^(E-2p). Smaller elements keep an absolute error of at
// most 2^(E-16). Token t's pieces are the B rows 8t..8t+7 of one MMA, and the
// epilogue adds the eight fp32 accumulator columns of each token.
//
// Work split: the rows are cut into groups of `rows` (a multiple of 8) rows,
// one group per CTA, or per cluster of 2 CTAs that split K in halves (rank 1
// hands its fp32 sums to rank 0 through distributed shared memory: rank 0's
// half first, then rank 1's). A group is walked in tiles of up to 128 rows
// (the MMA's M). A tile shorter than 128 rows still feeds 128 rows to the
// MMA: the rows past its end are whatever shared memory holds there, and
// only their own accumulator lanes, which are never read, depend on them.
// So a group needs no multiple of 128 rows and the groups fill the SMs.
//
// One CTA per group member, warp-specialised:
//   warps 0-3  epilogue and weight scales: per (tile, stage) warp q copies
//              the 16 E8M0 bytes of stage rows 32q..32q+31 (cp.async, a few
//              items ahead) into its TMEM quarter; per batch of tiles,
//              accumulators -> y.
//   warp 4     TMA producer: one 3D copy per (tile, stage) of 2 atoms of 256
//              K values x the tile's rows, L2 evict-first.
//   warp 5     MMA issuer (one thread) and TMEM owner: 8 MMAs of 128 x NPAD x
//              64 per (tile, stage); tcgen05.commit frees the buffers.
//   warps 6-13 converters, two groups of four: per stage (the groups take
//              turns), the activation pieces (swizzled for the MMA) and
//              their scale words (into TMEM, each warp its lane quarter).
// Every wait is bounded (device_common.cuh); on a timeout the status word is
// set and every role winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "f4_linear_launch.h"
#include "tc_common.cuh"

namespace mxfp4 {
namespace f4 {

using tc::commit_to;
using tc::fence_after_sync;
using tc::fence_before_sync;
using tc::operand_desc;

constexpr int kTileRows = 128;      // MMA M
constexpr int kStageK = 512;        // K values per stage (two atoms)
constexpr int kAtomRowBytes = 128;  // one atom of one row: 256 packed codes
constexpr int kEpilogueWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kFirstConverterWarp = 6;
// Converters: kGroups groups of kGroupWarps warps; group g converts stages
// g, g + kGroups, ..., so that many stages are converted at once (one warp
// alone is latency-bound on the conversion's dependent steps).
constexpr int kGroups = 2;
constexpr int kGroupWarps = 4;
constexpr int kConverters = kGroups * kGroupWarps;
constexpr int kThreads = (kFirstConverterWarp + kConverters) * 32;
constexpr int kMaxNA = 8;

// Weight scales run this many (tile, stage) items ahead of their use: each
// epilogue lane keeps a ring of 16-byte slots filled by cp.async (HBM
// latency would otherwise stall every item).
constexpr int kScaleAhead = 2;  // a power of two
static_assert((kScaleAhead & (kScaleAhead - 1)) == 0, "ring index by mask");
constexpr int kScaleRingBytes = kEpilogueWarps * kScaleAhead * 32 * 16;

// Shared-memory plan (offsets from the 1024-aligned base). The weight ring
// first: NA slots of 2 atoms x h_main rows x 128 B. The MMA reads 128 rows
// of an atom whatever the tile's height, i.e. up to (128 - h_main) x 128
// bytes past the ring's last atom; those rows' results are never read, and
// what lies there is the next region, so no slack is needed while the
// allocation reaches that far. Then NB activation buffers of 2 atoms of
// NPAD rows x 128 B, their scale images (NPAD x 16 bytes: row n's 16 block
// scales of the stage), the mbarriers, the abort flag, the TMEM base word,
// the cluster inbox and the epilogue warps' weight-scale rings.
template <int NPAD>
struct Layout {
    static constexpr int kAtomBytesB = NPAD * kAtomRowBytes;
    static constexpr int kSlotB = 2 * kAtomBytesB;  // a multiple of 1024 (NPAD >= 16)
    static constexpr int kImgBytes = NPAD * 16;
    static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 128, "MMA N");
    static_assert(kSlotB % 1024 == 0, "B buffers stay 1024-aligned for the 128-byte swizzle");

    // Runtime part (depends on NA, NB, the cluster inbox and h_main).
    int slot_a, off_b, off_img, off_bars, off_abort, off_tmem_slot, off_inbox, off_sc, total;
    __host__ __device__ Layout(int na, int nb, int inbox_bytes, int h_main) {
        slot_a = 2 * h_main * kAtomRowBytes;  // a multiple of 2048 (h_main % 8 == 0)
        off_b = na * slot_a;
        off_img = off_b + nb * kSlotB;
        off_bars = off_img + nb * kImgBytes;
        const int nbars = 3 * na + 3 * nb + 4;
        off_abort = off_bars + 8 * nbars;
        off_tmem_slot = off_abort + 4;
        off_inbox = (off_tmem_slot + 4 + 127) / 128 * 128;
        off_sc = (off_inbox + inbox_bytes + 127) / 128 * 128;
        total = off_sc + kScaleRingBytes;
        const int a_reach = off_b + (kTileRows - h_main) * kAtomRowBytes;
        total = total > a_reach ? total : a_reach;
    }
};

struct Bars {
    uint32_t base;
    int na, nb;
    __device__ uint32_t full_a(int s) const { return base + 8 * s; }
    __device__ uint32_t empty_a(int s) const { return base + 8 * (na + s); }
    __device__ uint32_t sfa_ready(int s) const { return base + 8 * (2 * na + s); }
    __device__ uint32_t full_b(int s) const { return base + 8 * (3 * na + s); }
    __device__ uint32_t empty_b(int s) const { return base + 8 * (3 * na + nb + s); }
    __device__ uint32_t img_ready(int s) const { return base + 8 * (3 * na + 2 * nb + s); }
    __device__ uint32_t acc_full() const { return base + 8 * (3 * na + 3 * nb); }
    __device__ uint32_t acc_empty() const { return base + 8 * (3 * na + 3 * nb + 1); }
    __device__ uint32_t inbox() const { return base + 8 * (3 * na + 3 * nb + 2); }
    __device__ uint32_t drain() const { return base + 8 * (3 * na + 3 * nb + 3); }
};

// The CTA's share: tiles [0, ntile) of its group (row r0 + 128 i; the last
// tile of a group with a tail is h_tail rows), in batches of sizes as even as
// possible; K stages [st0, st0 + spt).
struct Work {
    int r0, ntile, nbatch;
    int st0, spt;
    uint32_t rank;
    int tail_tile;  // index of the tail tile, or -1
    __device__ int batch_begin(int b) const { return ntile * b / nbatch; }
    __device__ int batch_size(int b) const { return ntile * (b + 1) / nbatch - ntile * b / nbatch; }
    __device__ int tile_row0(int i) const { return r0 + i * kTileRows; }
};

__device__ __forceinline__ int tile_height(const F4Params& p, const Work& w, int i) {
    return i == w.tail_tile ? p.h_tail : p.h_main;
}

// Ring position: slot index and the parity of its current round.
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ void next(int n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// The two halves of a cluster barrier (every thread of every CTA arrives,
// then waits before its next arrival).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// ------------------------------------------------------------- producer
__device__ void producer(const F4Params& p, const CUtensorMap* main_map, const CUtensorMap* tail_map, const Work& w,
                         uint32_t a_base, int slot_a, const Bars& bars, const WaitCtx& wc) {
    const uint64_t policy = l2_evict_first_policy();
    asm volatile("prefetch.tensormap [%0];" ::"l"(main_map) : "memory");
    if (w.tail_tile >= 0) asm volatile("prefetch.tensormap [%0];" ::"l"(tail_map) : "memory");
    const int na = p.na;
    Ring r;
    int issued = 0;
    bool ok = true;
    for (int b = 0; b < w.nbatch && ok; ++b) {
        const int t0 = w.batch_begin(b), bt = w.batch_size(b);
        for (int k = 0; k < w.spt && ok; ++k) {
            const int atom0 = (w.st0 + k) * 2;
            for (int ti = t0; ti < t0 + bt; ++ti) {
                if (!mbar_wait(bars.empty_a(r.slot), r.phase ^ 1u, wc)) {
                    ok = false;
                    break;
                }
                const uint32_t slot = a_base + r.slot * slot_a;
                if (withhold_stage(static_cast<uint32_t>(issued))) {  // test-only builds
                    ++issued;
                    r.next(na);
                    continue;
                }
                const bool tail = ti == w.tail_tile;
                const int h = tail ? p.h_tail : p.h_main;
                mbar_arrive_expect_tx(bars.full_a(r.slot), static_cast<uint32_t>(2 * h * kAtomRowBytes));
                tma_load_3d(slot, tail ? tail_map : main_map, 0, w.tile_row0(ti), atom0, bars.full_a(r.slot), policy);
                ++issued;
                r.next(na);
            }
        }
    }
    if (!ok) {
        // Let the copies in flight land (bounded, whatever the abort flag
        // says) before the CTA may exit.
        int never = 0;
        const WaitCtx own{p.status, &never};
        for (int j = issued > na ? issued - na : 0; j < issued; ++j)
            mbar_wait(bars.full_a(j % na), static_cast<uint32_t>((j / na) & 1), own);
    }
}

// ----------------------------------------------------------- MMA issuer
// Per (tile, stage): 8 MMAs of K = 64. MMA m of the stage reads atom m / 4 at
// byte 32 (m % 4) of each row, and the scale word m / 2 of its buffer (4
// columns apart), bytes 2 (m % 2) and 2 (m % 2) + 1 (scale ID 0 or 2).
template <int NPAD>
__device__ bool mma_issue_all(const F4Params& p, const Work& w, uint32_t a_base, int slot_a, uint32_t b_base,
                              uint32_t tbase, uint32_t sfa_col, uint32_t sfb_col, const Bars& bars,
                              const WaitCtx& wc) {
    using L = Layout<NPAD>;
    const int na = p.na;
    const uint32_t id0 = tc::mma_idesc(tc::kFmtMxf4E2M1, tc::kFmtMxf4E2M1, kTileRows, NPAD, 0);
    const uint32_t id2 = tc::mma_idesc(tc::kFmtMxf4E2M1, tc::kFmtMxf4E2M1, kTileRows, NPAD, 2);
    Ring ra, rb;
    for (int b = 0; b < w.nbatch; ++b) {
        const int t0 = w.batch_begin(b), bt = w.batch_size(b);
        if (!mbar_wait(bars.acc_empty(), (static_cast<uint32_t>(b) & 1u) ^ 1u, wc)) return false;
        for (int k = 0; k < w.spt; ++k) {
            const uint64_t bd = operand_desc(b_base + rb.slot * L::kSlotB);
            const uint32_t sfb = tbase + sfb_col + rb.slot * 16;
            for (int ti = t0; ti < t0 + bt; ++ti) {
                // The stage's activations (first tile only), the tile's
                // weights and its scale words: all tested at once, and waited
                // for one by one (bounded) only if some are not there yet.
                const bool ready = ti == t0 ? mbar_test3(bars.full_b(rb.slot), rb.phase, bars.full_a(ra.slot), ra.phase,
                                                         bars.sfa_ready(ra.slot), ra.phase)
                                            : mbar_test2(bars.full_a(ra.slot), ra.phase, bars.sfa_ready(ra.slot), ra.phase);
                if (!ready) {
                    if (ti == t0 && !mbar_wait(bars.full_b(rb.slot), rb.phase, wc)) return false;
                    if (!mbar_wait(bars.full_a(ra.slot), ra.phase, wc)) return false;
                    if (!mbar_wait(bars.sfa_ready(ra.slot), ra.phase, wc)) return false;
                }
                fence_after_sync();
                const uint64_t ad = operand_desc(a_base + ra.slot * slot_a);
                const uint32_t atom_a = static_cast<uint32_t>(tile_height(p, w, ti) * kAtomRowBytes);
                const uint32_t sfa = tbase + sfa_col + ra.slot * 16;
                const uint32_t d_tmem = tbase + (ti - t0) * NPAD;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const uint32_t off_a = (m >> 2) * atom_a + 32 * (m & 3);
                    const uint32_t off_b = (m >> 2) * L::kAtomBytesB + 32 * (m & 3);
                    tc::mma_mxf4(d_tmem, ad + (off_a >> 4), bd + (off_b >> 4), (m & 1) ? id2 : id0, sfa + 4 * (m >> 1),
                                 sfb + 4 * (m >> 1), (m | k) != 0);
                }
                commit_to(bars.empty_a(ra.slot));
                ra.next(na);
            }
            commit_to(bars.empty_b(rb.slot));
            rb.next(p.nb);
        }
        commit_to(bars.acc_full());
    }
    return true;
}

template <int NPAD>
__device__ void mma_issuer(const F4Params& p, const Work& w, uint32_t a_base, int slot_a, uint32_t b_base,
                           uint32_t tbase, uint32_t sfa_col, uint32_t sfb_col, const Bars& bars, const WaitCtx& wc) {
    if (mma_issue_all<NPAD>(p, w, a_base, slot_a, b_base, tbase, sfa_col, sfb_col, bars, wc)) return;
    // Aborted: MMAs issued so far may still read shared memory and write
    // TMEM. One more commit tracks them all; wait for it (bounded, whatever
    // the abort flag says) before the CTA frees TMEM and exits.
    commit_to(bars.drain());
    int never = 0;
    const WaitCtx own{wc.status, &never};
    mbar_wait(bars.drain(), 0, own);
}

// ------------------------------------------------------------ converter
// The eight 2-bit digits of a 16-bit X, digit j moved to bits 4j and 4j + 1.
__device__ __forceinline__ uint32_t spread_digits(uint32_t x) {
    x = (x | (x << 8)) & 0x00FF00FFu;
    x = (x | (x << 4)) & 0x0F0F0F0Fu;
    return (x | (x << 2)) & 0x33333333u;
}

// Transpose of an 8 x 8 matrix of nibbles: on entry word i holds row i
// (nibble j = column j); on exit word j holds column j (nibble i = row i).
// Three rounds: 16-bit halves between words 4 apart, bytes between words 2
// apart, nibbles between neighbours.
__device__ __forceinline__ void transpose_nibbles(uint32_t (&s)[8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = s[i], b = s[i + 4];
        s[i] = prmt(a, b, 0x5410);
        s[i + 4] = prmt(a, b, 0x7632);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 4 * h; i < 4 * h + 2; ++i) {
            const uint32_t a = s[i], b = s[i + 2];
            s[i] = prmt(a, b, 0x6240);
            s[i + 2] = prmt(a, b, 0x7351);
        }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint32_t a = s[i], b = s[i + 1];
        s[i] = (a & 0x0F0F0F0Fu) | ((b & 0x0F0F0F0Fu) << 4);
        s[i + 1] = ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
    }
}

// Stores the 4-byte word of piece P of a lane's 8 elements: B row 8t + P
// (row % 8 == P), swizzled 16-byte chunk blk ^ P. With base = row 8t's
// address plus blk << 4 (bits 4-6) and 4j, the address is one XOR of bits
// 4-6 and an immediate row offset.
template <int P>
__device__ __forceinline__ void store_piece(uint32_t base, uint32_t v) {
    asm volatile("st.shared.u32 [%0+%2], %1;" ::"r"(base ^ (P << 4)), "r"(v), "n"(P * 128) : "memory");
}

// One element pair's digit words: X of elements 2q and 2q + 1 in the low
// 16 bits of x2.x and x2.y; sg0 / sg1 hold each element's sign bit copied
// into bit 7 of every byte. Word i gets element i's eight 2-bit digits,
// digit d in bits 4d and 4d + 1, the sign in bit 4d + 3: the bytes of X go
// to 16-bit halves (one byte permute), then to nibbles, then to 2-bit
// fields.
__device__ __forceinline__ void digit_words(float2 x2, uint32_t sg0, uint32_t sg1, uint32_t& w0, uint32_t& w1) {
    uint32_t d0 = prmt(__float_as_uint(x2.x), 0u, 0x4140);
    uint32_t d1 = prmt(__float_as_uint(x2.y), 0u, 0x4140);
    d0 = (d0 | (d0 << 4)) & 0x0F0F0F0Fu;
    d1 = (d1 | (d1 << 4)) & 0x0F0F0F0Fu;
    d0 = (d0 | (d0 << 2)) & 0x33333333u;
    d1 = (d1 | (d1 << 2)) & 0x33333333u;
    w0 = d0 | (sg0 & 0x88888888u);
    w1 = d1 | (sg1 & 0x88888888u);
}

// Writes one unit (token t): after the transpose, the lane's word of each of
// the token's 8 piece rows of the swizzled B atom (piece p is digit 7 - p),
// and the scale bytes E - 2p + 127 of pieces 2j and 2j + 1 (image row
// 8t + p, byte sbyte0).
__device__ __forceinline__ void emit_unit(uint32_t (&s)[8], int e, int t, int blk, int j, uint32_t atom,
                                          uint32_t img, int sbyte0) {
    transpose_nibbles(s);  // s[d]: digit d, element i in nibble i
    const uint32_t base = atom + static_cast<uint32_t>(t) * 1024u + 4u * static_cast<uint32_t>(j) +
                          (static_cast<uint32_t>(blk) << 4);
    store_piece<0>(base, s[7]);
    store_piece<1>(base, s[6]);
    store_piece<2>(base, s[5]);
    store_piece<3>(base, s[4]);
    store_piece<4>(base, s[3]);
    store_piece<5>(base, s[2]);
    store_piece<6>(base, s[1]);
    store_piece<7>(base, s[0]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int p = 2 * j + h;
        const uint32_t ad = img + static_cast<uint32_t>((8 * t + p) * 16 + sbyte0);
        asm volatile("st.shared.u8 [%0], %1;" ::"r"(ad), "r"(static_cast<uint32_t>(e - 2 * p + 127)) : "memory");
    }
}

// The block exponent E from the largest magnitude's exponent field (0 for
// zero and subnormal blocks), at least -112 so that every piece scale
// 2^(E - 2p) is a valid E8M0 value (byte >= 1); returned with the factor
// 2^(15 - E) (exponent field in [14, 254]). X = rne(|x| 2^(15-E)) < 2^16
// then lands in the low mantissa bits of |x| 2^(15-E) + 1.5 * 2^23 (one
// rounding: the product is exact).
__device__ __forceinline__ int block_exponent(int field, float& f) {
    const int e = max(field - 127, -112);
    f = __int_as_float((142 - e) << 23);
    return e;
}

// One unit of bf16 activations: a lane's 8 consecutive values of a 32-value
// block (one 16-byte load; word q holds elements 2q (low half) and 2q + 1),
// token t; the block is held by the 4 lanes l with l >> 2 == blk (j = l & 3
// holds elements 8j..8j+7).
__device__ __forceinline__ void convert_unit(const uint4& v, int t, int blk, int j, uint32_t atom, uint32_t img,
                                             int sbyte0) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) a[q] = w[q] & 0x7fff7fffu;
    const uint32_t m = __vmaxu2(__vmaxu2(a[0], a[1]), __vmaxu2(a[2], a[3]));
    uint32_t amax = max(m & 0xffffu, m >> 16);
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    float f;
    const int e = block_exponent(static_cast<int>(amax >> 7), f);
    const uint64_t f2 = f32x2_pack(f, f), c2 = f32x2_pack(12582912.0f, 12582912.0f);
    uint32_t s[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 x2 = f32x2_unpack(
            f32x2_fma(f32x2_pack(__uint_as_float(a[q] << 16), __uint_as_float(a[q] & 0xffff0000u)), f2, c2));
        // The permute's sign mode copies bit 15 (byte 1) or bit 31 (byte 3).
        digit_words(x2, prmt(w[q], 0u, 0x9999), prmt(w[q], 0u, 0xBBBB), s[2 * q], s[2 * q + 1]);
    }
    emit_unit(s, e, t, blk, j, atom, img, sbyte0);
}

// The same for 8 fp32 values (elements 0..7 of the lane's share).
__device__ __forceinline__ void convert_unit_f32(const float (&h)[8], int t, int blk, int j, uint32_t atom,
                                                 uint32_t img, int sbyte0) {
    uint32_t a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = __float_as_uint(h[i]) & 0x7fffffffu;
    uint32_t amax = max(max(max(a[0], a[1]), max(a[2], a[3])), max(max(a[4], a[5]), max(a[6], a[7])));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    float f;
    const int e = block_exponent(static_cast<int>(amax >> 23), f);
    const uint64_t f2 = f32x2_pack(f, f), c2 = f32x2_pack(12582912.0f, 12582912.0f);
    uint32_t s[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 x2 =
            f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(a[2 * q]), __uint_as_float(a[2 * q + 1])), f2, c2));
        digit_words(x2, prmt(__float_as_uint(h[2 * q]), 0u, 0xBBBB), prmt(__float_as_uint(h[2 * q + 1]), 0u, 0xBBBB),
                    s[2 * q], s[2 * q + 1]);
    }
    emit_unit(s, e, t, blk, j, atom, img, sbyte0);
}

// Converter groups. Group g converts stages g, g + kGroups, ...; warp m of
// the group converts units (token t, atom c) m, m + 4, ... of the stage's 2T
// (a unit is 8 blocks of 32 values, 4 lanes per block; at most NPAD / 16
// units a warp). Each stage's x loads are issued two of the group's stages
// ahead, and positions advance by counting (no division per stage). The four
// warps of a group lie in the four TMEM lane quarters (warp % 4), so once
// the stage's scale image is complete (img_ready) each stores the piece
// scale words into its own quarter, then hands the stage to the MMA
// (full_b).
struct StageCursor {
    int left;        // the group's stages still to visit
    int k;           // K stage of the current stage (st0 .. st0 + spt - 1)
    int slot;        // B buffer of the current stage
    uint32_t phase;  // parity of the buffer's current use
    __device__ void next(int st0, int spt, int nb) {
        --left;
        k += kGroups;
        while (k >= st0 + spt) k -= spt;
        slot += kGroups;
        while (slot >= nb) {
            slot -= nb;
            phase ^= 1u;
        }
    }
};

// Piece scale words into one warp's 32 lanes. Each 32-row quarter of the MMA
// reads the B scales from its own lanes: B row n at lane n % 32, column
// (scale address + n / 32); so every warp stores word a of B rows l + 32i
// (vi, i < 4) at column 4a + i.
__device__ __forceinline__ void store_b_scale_words(uint32_t taddr, const uint4& v0, const uint4& v1,
                                                    const uint4& v2, const uint4& v3) {
    const uint32_t c16[16] = {v0.x, v1.x, v2.x, v3.x, v0.y, v1.y, v2.y, v3.y,
                              v0.z, v1.z, v2.z, v3.z, v0.w, v1.w, v2.w, v3.w};
    tc::tmem_store16(taddr, c16);
    tc::tmem_wait_st();
    fence_before_sync();
}

// IN = 0: x is bf16 [T, K]. IN = 1: x[t, k] = SiLU(a) * b in fp32 with
// a = xab[t, k] and b = xab[t, K + k] (rows of 2K floats), a 32-byte load
// of each per unit and 8 fp32 values converted.
template <int NPAD, int IN>
__device__ void converter(const F4Params& p, int cw, int warp, int lane, const Work& w, uint32_t b_base,
                          uint32_t img_base, uint32_t tbase, uint32_t sfb_col, const Bars& bars, const WaitCtx& wc) {
    using L = Layout<NPAD>;
    constexpr int NU = NPAD / 16;
    constexpr int NW = IN ? 4 : 1;  // 16-byte loads per unit
    const int g = cw / kGroupWarps, m = cw % kGroupWarps;
    const int nst = w.nbatch * w.spt;
    const int nstg = nst > g ? (nst - g + kGroups - 1) / kGroups : 0;
    if (nstg == 0) return;
    pdl_wait_previous();  // x may come from the previous kernel of the stream
    const int nb = p.nb;
    StageCursor cur{nstg, w.st0 + g % w.spt, g % nb, static_cast<uint32_t>((g / nb) & 1)};
    StageCursor ld = cur;
    const int blk = lane >> 2, jj = lane & 3;
    const __nv_bfloat16* xl = IN == 0 ? p.x + blk * 32 + 8 * jj : nullptr;
    const float* xf = IN == 1 ? p.xab + blk * 32 + 8 * jj : nullptr;
    const uint32_t lanes = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int nun = m < 2 * p.T ? (2 * p.T - m + kGroupWarps - 1) / kGroupWarps : 0;  // units of this warp
    auto load = [&](StageCursor& c, uint4 (&v)[NU][NW]) {
        if (c.left <= 0) return;
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int unit = m + kGroupWarps * u;
            // Through L2 only: x may have been written by the previous kernel
            // of the stream, which this kernel overlaps.
            if (unit >= 2 * p.T) continue;
            const size_t off = static_cast<size_t>(c.k) * kStageK + (unit & 1) * 256;
            if (IN == 0) {
                v[u][0] = __ldcg(reinterpret_cast<const uint4*>(xl + static_cast<size_t>(unit >> 1) * p.K + off));
            } else {
                const float* a = xf + static_cast<size_t>(unit >> 1) * 2 * p.K + off;
                v[u][0] = __ldcg(reinterpret_cast<const uint4*>(a));
                v[u][NW > 1 ? 1 : 0] = __ldcg(reinterpret_cast<const uint4*>(a + 4));
                v[u][NW > 2 ? 2 : 0] = __ldcg(reinterpret_cast<const uint4*>(a + p.K));
                v[u][NW > 3 ? 3 : 0] = __ldcg(reinterpret_cast<const uint4*>(a + p.K + 4));
            }
        }
        c.next(w.st0, w.spt, nb);
    };
    auto stage = [&](const uint4 (&v)[NU][NW]) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(bars.empty_b(cur.slot), cur.phase ^ 1u, wc))) return false;
        const uint32_t bslot = b_base + cur.slot * L::kSlotB;
        const uint32_t img = img_base + cur.slot * L::kImgBytes;
        // Units m + 4u: atom c = m & 1 for all of them, tokens m / 2 + 2u;
        // one after the other (in isolation two units in lockstep measured
        // 676 cycles against 2 x 290 one at a time).
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            if (u >= nun) break;
            const uint32_t atom = bslot + (m & 1) * L::kAtomBytesB;
            if (IN == 0) {
                convert_unit(v[u][0], (m >> 1) + 2 * u, blk, jj, atom, img, 8 * (m & 1) + blk);
            } else {
                const uint4 a0 = v[u][0], a1 = v[u][NW > 1 ? 1 : 0], b0 = v[u][NW > 2 ? 2 : 0],
                            b1 = v[u][NW > 3 ? 3 : 0];
                const uint32_t av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                const uint32_t bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                float h[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    // SiLU(a) * b with the hardware exponential and
                    // reciprocal: a few ulp of fp32, far below the 16 bits
                    // below the block maximum that the pieces keep. a very
                    // negative: 1 + e^-a is inf and the quotient 0.
                    const float a = __uint_as_float(av[i]);
                    h[i] = __fdividef(a, 1.0f + __expf(-a)) * __uint_as_float(bv[i]);
                }
                convert_unit_f32(h, (m >> 1) + 2 * u, blk, jj, atom, img, 8 * (m & 1) + blk);
            }
        }
        fence_proxy_async_shared();  // this warp's piece writes -> visible to the tensor core's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.img_ready(cur.slot));
        if (!__all_sync(0xffffffffu, mbar_wait(bars.img_ready(cur.slot), cur.phase, wc))) return false;
        const uint4 v0 = lds128(img + lane * 16);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint4 v1 = lane + 32 < NPAD ? lds128(img + (lane + 32) * 16) : z;
        const uint4 v2 = lane + 64 < NPAD ? lds128(img + (lane + 64) * 16) : z;
        const uint4 v3 = lane + 96 < NPAD ? lds128(img + (lane + 96) * 16) : z;
        store_b_scale_words(tbase + lanes + sfb_col + cur.slot * 16, v0, v1, v2, v3);
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.full_b(cur.slot));
        cur.next(w.st0, w.spt, nb);
        return true;
    };
    uint4 va[NU][NW], vb[NU][NW];
    load(ld, va);
    load(ld, vb);
    while (cur.left > 0) {
        if (!stage(va)) return;
        load(ld, va);
        if (cur.left <= 0) break;
        if (!stage(vb)) return;
        load(ld, vb);
    }
}

// ------------------------------------------------------------- epilogue
// Weight scale words of one buffer into warp q's 32 lanes: word a (blocks
// 4a..4a+3 of the stage) at column 4a + q, where the MMA reads row r's word
// (lane r, column scale address + r / 32).
__device__ __forceinline__ void store_a_scale_words(uint32_t taddr, int q, const uint4& v) {
    uint32_t c16[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) c16[i] = 0u;
    switch (q) {  // warp-uniform
        case 0: c16[0] = v.x; c16[4] = v.y; c16[8] = v.z; c16[12] = v.w; break;
        case 1: c16[1] = v.x; c16[5] = v.y; c16[9] = v.z; c16[13] = v.w; break;
        case 2: c16[2] = v.x; c16[6] = v.y; c16[10] = v.z; c16[14] = v.w; break;
        default: c16[3] = v.x; c16[7] = v.y; c16[11] = v.z; c16[15] = v.w; break;
    }
    tc::tmem_store16(taddr, c16);
    tc::tmem_wait_st();
    fence_before_sync();
}

// 16-byte vectors per inbox row: the tokens' sums (NPAD / 8 of them) in
// groups of 4.
__host__ __device__ constexpr int inbox_vectors(int npad) { return (npad / 8 + 3) / 4; }

// Asynchronous store of 16 bytes into a peer CTA's shared memory, counted
// as transaction bytes on the peer's mbarrier (cluster addresses).
__device__ __forceinline__ void st_async_v4(uint32_t dst, float a, float b, float c, float d, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(dst),
                 "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
                 : "memory");
}

// 16-byte global -> shared copy through L2 on the load/store path; with
// src_bytes = 0 it writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most kScaleAhead - 1 of this thread's copy groups are pending.
__device__ __forceinline__ void cp_async_wait_ahead() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kScaleAhead - 1) : "memory");
}

// Requests the weight scales of the (tile, stage) items in streaming order
// (batch, stage, tile), one lane's row each, into the lane's ring (slots 512
// bytes apart): item i lands in slot i % kScaleAhead as copy group i (one
// group per item, empty past the last item, so group counts stay aligned
// with items).
struct ScaleFeed {
    int b = 0, k = 0, ti = 0;
    int t0 = 0, t1 = 0;  // the current batch's tiles [t0, t1)
    int issued = 0;
    __device__ void start(const Work& w) {
        t0 = ti = w.batch_begin(0);
        t1 = t0 + w.batch_size(0);
    }
    __device__ void request(const F4Params& p, const Work& w, int rt, uint32_t ring) {
        if (b < w.nbatch) {
            const int row = w.tile_row0(ti) + rt;
            const bool ok = rt < tile_height(p, w, ti) && row < p.N;
            const uint8_t* src = ok ? p.ws + static_cast<size_t>(row) * p.nblk + static_cast<size_t>(w.st0 + k) * 16
                                    : p.ws;
            cp_async16(ring + (issued & (kScaleAhead - 1)) * 512, src, ok ? 16u : 0u);
            if (++ti == t1) {
                ti = t0;
                if (++k == w.spt) {
                    k = 0;
                    if (++b < w.nbatch) {
                        t0 = ti = w.batch_begin(b);
                        t1 = t0 + w.batch_size(b);
                    }
                }
            }
        }
        cp_async_commit();
        ++issued;
    }
};

// Warp q of the epilogue group: per (tile, stage) the weight scale words of
// tile rows 32q..32q+31, per stage the piece scale words, per batch the
// accumulators -> y (lane = tile row 32q + lane; token t = the sum of
// columns 8t..8t+7, smallest piece first).
template <int NPAD>
__device__ void epilogue_body(const F4Params& p, int q, int lane, const Work& w, uint32_t inbox, uint32_t sc_ring,
                              uint32_t tbase, uint32_t sfa_col, const Bars& bars,
                              const WaitCtx& wc, bool& cluster_waited) {
    const int T = p.T, na = p.na;
    bool waited = false;  // for the previous kernel of the stream (before the first write of y)
    const int rt = q * 32 + lane;
    const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
    // The lane's ring: kScaleAhead slots of 16 bytes, 512 bytes apart per
    // slot (lanes side by side). Weights and scales do not come from the
    // previous kernel, so the requests start at once.
    const uint32_t ring = sc_ring + static_cast<uint32_t>(q * kScaleAhead * 512 + lane * 16);
    ScaleFeed feed;
    feed.start(w);
    for (int d = 0; d < kScaleAhead; ++d) feed.request(p, w, rt, ring);
    int used = 0;
    Ring ra;
    for (int b = 0; b < w.nbatch; ++b) {
        const int t0 = w.batch_begin(b), bt = w.batch_size(b);
        // Items come in the feed's order; rows past the tile or past N have
        // zero scales.
        auto weight_scales = [&](int, int) -> bool {
            cp_async_wait_ahead();
            const uint4 v = lds128(ring + (used & (kScaleAhead - 1)) * 512);
            ++used;
            feed.request(p, w, rt, ring);
            // The buffer's TMEM columns are free once the MMAs of the item
            // NA back have completed (their commit).
            if (!__all_sync(0xffffffffu, mbar_wait(bars.empty_a(ra.slot), ra.phase ^ 1u, wc))) return false;
            fence_after_sync();
            store_a_scale_words(tbase + lanes + sfa_col + ra.slot * 16, q, v);
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.sfa_ready(ra.slot));
            ra.next(na);
            return true;
        };
        for (int k = 0; k < w.spt; ++k)
            for (int ti = t0; ti < t0 + bt; ++ti)
                if (!weight_scales(k, ti)) return;
        if (!__all_sync(0xffffffffu, mbar_wait(bars.acc_full(), static_cast<uint32_t>(b) & 1u, wc))) return;
        fence_after_sync();
        if (!waited) {
            pdl_wait_previous();  // the previous kernel may still read y
            waited = true;
        }
        const bool sender = p.cl > 1 && w.rank != 0;
        if (p.cl > 1 && !cluster_waited) {
            cluster_wait();  // the peer has started (its barriers are initialised)
            cluster_waited = true;
        }
        if (p.cl > 1 && !sender) {
            // One batch per group when K is split: rank 1's sums of every
            // tile arrive together, counted in bytes on the inbox barrier.
            if (!__all_sync(0xffffffffu, mbar_wait(bars.inbox(), 0, wc))) return;
        }
        for (int ti = t0; ti < t0 + bt; ++ti) {
            // 16 accumulator columns (two tokens) at a time keeps the
            // registers down.
            float s[NPAD / 8];
#pragma unroll
            for (int c = 0; c < NPAD / 16; ++c) {
                uint32_t r[16];
                tc::tmem_load<16>(tbase + lanes + (ti - t0) * NPAD + 16 * c, r);
                tc::tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float a = __uint_as_float(r[8 * h + 7]);
#pragma unroll
                    for (int pc = 6; pc >= 0; --pc) a += __uint_as_float(r[8 * h + pc]);
                    s[2 * c + h] = a;
                }
            }
            // Inbox row of (tile, row), rows of the tile only (every tile
            // before the last has h_main): the sums of tokens 4v..4v+3 in
            // its 16-byte vector v.
            constexpr int NV = inbox_vectors(NPAD);
            const uint32_t row_off = static_cast<uint32_t>(((ti - t0) * p.h_main + rt) * NV * 16);
            if (sender) {
                if (rt >= tile_height(p, w, ti)) continue;
                // Hand the fp32 sums to rank 0: asynchronous remote stores
                // that count their bytes on rank 0's inbox barrier.
                const uint32_t dst = map_to_rank(inbox, 0) + row_off;
                const uint32_t rbar = map_to_rank(bars.inbox(), 0);
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    st_async_v4(dst + 16 * v, s[4 * v], 4 * v + 1 < NPAD / 8 ? s[4 * v + 1] : 0.f,
                                4 * v + 2 < NPAD / 8 ? s[4 * v + 2] : 0.f, 4 * v + 3 < NPAD / 8 ? s[4 * v + 3] : 0.f,
                                rbar);
                continue;
            }
            if (p.cl > 1 && rt < tile_height(p, w, ti)) {
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const uint4 in = lds128(inbox + row_off + 16 * v);
                    const float f4v[4] = {__uint_as_float(in.x), __uint_as_float(in.y), __uint_as_float(in.z),
                                          __uint_as_float(in.w)};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * v + e < NPAD / 8) s[4 * v + e] += f4v[e];
                }
            }
            const int row = w.tile_row0(ti) + rt;
            if (rt < tile_height(p, w, ti) && row < p.N) {
#pragma unroll
                for (int t = 0; t < NPAD / 8; ++t) {
                    if (t >= T) continue;
                    const size_t o = static_cast<size_t>(t) * p.N + row;
                    if (p.yf)
                        p.yf[o] = s[t];
                    else
                        p.y[o] = __float2bfloat16_rn(s[t]);
                }
            }
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.acc_empty());
    }
}

// On every way out (a timeout included) the lane's scale copies have landed
// before the CTA may exit.
template <int NPAD>
__device__ void epilogue(const F4Params& p, int q, int lane, const Work& w, uint32_t inbox, uint32_t sc_ring,
                         uint32_t tbase, uint32_t sfa_col, const Bars& bars,
                         const WaitCtx& wc, bool& cluster_waited) {
    epilogue_body<NPAD>(p, q, lane, w, inbox, sc_ring, tbase, sfa_col, bars, wc, cluster_waited);
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// --------------------------------------------------------------- kernel
// Up to 32 MMA columns (t <= 4) two CTAs share an SM (at most 72
// registers a thread); wider ones run one CTA per SM.
template <int NPAD, int IN>
__global__ void __launch_bounds__(kThreads, NPAD <= 32 && IN == 0 ? 2 : 1)
    f4_linear_kernel(const __grid_constant__ CUtensorMap main_map, const __grid_constant__ CUtensorMap tail_map,
                     const F4Params p) {
    using L = Layout<NPAD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();
    const L lay(p.na, p.nb, p.inbox_bytes, p.h_main);

    Work w;
    w.rank = p.cl > 1 ? cluster_ctarank() : 0u;
    const int group = p.cl > 1 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    w.r0 = group * p.rows;
    // Tiles of a whole group: one of h_main = rows when rows <= 128, else
    // rows / 128 of 128 rows and a tail tile of h_tail rows. The last group
    // keeps only the tiles that start below N (TMA fills rows past N with
    // zeros; their outputs are not written).
    const int full_tiles = p.rows <= kTileRows ? 1 : p.rows / kTileRows + (p.h_tail ? 1 : 0);
    const int in_n = p.N - w.r0;
    w.ntile = in_n > 0 ? min(full_tiles, (in_n + kTileRows - 1) / kTileRows) : 0;
    w.tail_tile = p.h_tail ? full_tiles - 1 : -1;
    w.nbatch = (w.ntile + p.max_batch - 1) / p.max_batch;
    w.st0 = p.stages * static_cast<int>(w.rank) / p.cl;
    w.spt = p.stages * (static_cast<int>(w.rank) + 1) / p.cl - w.st0;

    const Bars bars{base + static_cast<uint32_t>(lay.off_bars), p.na, p.nb};
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + lay.off_abort);
    const WaitCtx wc{p.status, abort_flag};
    const uint32_t tslot = base + lay.off_tmem_slot;

    if (warp == kMmaWarp) {
        tc::tmem_alloc(tslot, static_cast<uint32_t>(p.tmem_cols));
        tc::tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        for (int s = 0; s < p.na; ++s) {
            mbar_init(bars.full_a(s), 1);
            mbar_init(bars.empty_a(s), 1);
            mbar_init(bars.sfa_ready(s), kEpilogueWarps);
        }
        for (int s = 0; s < p.nb; ++s) {
            mbar_init(bars.full_b(s), kGroupWarps);
            mbar_init(bars.empty_b(s), 1);
            mbar_init(bars.img_ready(s), kGroupWarps);
        }
        mbar_init(bars.acc_full(), 1);
        mbar_init(bars.acc_empty(), kEpilogueWarps);
        mbar_init(bars.inbox(), 1);
        mbar_init(bars.drain(), 1);
        *abort_flag = 0;
        fence_barrier_init();
        // Rank 0 of a cluster expects rank 1's sums of every row of its
        // tiles, in bytes (rank 1 sends only after the cluster barrier, so
        // this comes first).
        if (p.cl > 1 && w.rank == 0 && w.ntile > 0) {
            int rows = 0;
            for (int i = 0; i < w.ntile; ++i) rows += tile_height(p, w, i);
            mbar_arrive_expect_tx(bars.inbox(), static_cast<uint32_t>(rows * inbox_vectors(NPAD) * 16));
        }
    }
    // Rows past 8T of the B buffers (padding of the MMA's N) and their scale
    // bytes are zero for the whole kernel; the converters never write them.
    const int pad_rows = NPAD - 8 * p.T;
    if (pad_rows > 0) {
        const int chunks = p.nb * 2 * pad_rows * 8;  // 16-byte chunks: buffer, atom, row, chunk
        for (int i = threadIdx.x; i < chunks + p.nb * pad_rows; i += kThreads) {
            uint32_t a;
            if (i < chunks) {
                const int row = 8 * p.T + (i >> 3) % pad_rows, atom = (i >> 3) / pad_rows;  // atom over buffers
                a = base + lay.off_b + atom * L::kAtomBytesB + (row >> 3) * 1024 + (row & 7) * 128 + (i & 7) * 16;
            } else {
                const int r = i - chunks;
                a = base + lay.off_img + (r / pad_rows) * L::kImgBytes + (8 * p.T + r % pad_rows) * 16;
            }
            sts128(a, 0u, 0u, 0u, 0u);
        }
    }
    fence_proxy_async_shared();
    // Cluster: arrive now, wait only before the first access to the peer's
    // shared memory (the epilogue's hand-off) or at the end.
    if (p.cl > 1) cluster_arrive();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = lds_u32_volatile(tslot);
    // TMEM: accumulators from column 0 (NPAD per tile of a batch); scale
    // columns at the top, 16 per weight slot then 16 per activation buffer.
    const uint32_t sfa_col = static_cast<uint32_t>((p.tmem_cols - 16 * p.na - 16 * p.nb) / 32 * 32);
    const uint32_t sfb_col = sfa_col + 16u * static_cast<uint32_t>(p.na);
    const uint32_t a_base = base;

    bool cluster_waited = false;
    if (w.ntile > 0 && w.spt > 0) {
        if (warp == kProducerWarp) {
            if (lane == 0) producer(p, &main_map, &tail_map, w, a_base, lay.slot_a, bars, wc);
        } else if (warp == kMmaWarp) {
            if (lane == 0)
                mma_issuer<NPAD>(p, w, a_base, lay.slot_a, base + lay.off_b, tbase, sfa_col, sfb_col, bars, wc);
        } else if (warp >= kFirstConverterWarp) {
            converter<NPAD, IN>(p, warp - kFirstConverterWarp, warp, lane, w, base + lay.off_b, base + lay.off_img, tbase,
                            sfb_col, bars, wc);
        } else {
            epilogue<NPAD>(p, warp, lane, w, base + lay.off_inbox, base + lay.off_sc, tbase, sfa_col, bars, wc,
                           cluster_waited);
        }
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        fence_after_sync();
        tc::tmem_dealloc(tbase, static_cast<uint32_t>(p.tmem_cols));
    }
    // No CTA of a cluster leaves while a peer may still write to it.
    if (p.cl > 1) {
        if (!cluster_waited) cluster_wait();
        cluster_sync_all();
    }
}

// ----------------------------------------------------------------- host
template <int NPAD, int IN>
static cudaError_t launch_npad(const CUtensorMap& main_map, const CUtensorMap& tail_map, const F4Params& p,
                               const F4Plan& plan, cudaStream_t stream) {
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || configured[dev] < plan.smem_bytes) {
        cudaError_t e = cudaFuncSetAttribute(f4_linear_kernel<NPAD, IN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             plan.smem_bytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = plan.smem_bytes;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(kThreads);
    cfg.gridDim = dim3(plan.grid);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.cl > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = p.cl;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, f4_linear_kernel<NPAD, IN>, main_map, tail_map, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

static int npad_for(int t) { return t <= 2 ? 16 : (t <= 4 ? 32 : (t <= 6 ? 48 : (t <= 8 ? 64 : 128))); }

static int smem_layout_bytes(int npad, int na, int nb, int inbox, int h_main) {
    switch (npad) {
        case 16: return Layout<16>(na, nb, inbox, h_main).total;
        case 32: return Layout<32>(na, nb, inbox, h_main).total;
        case 48: return Layout<48>(na, nb, inbox, h_main).total;
        case 64: return Layout<64>(na, nb, inbox, h_main).total;
        default: return Layout<128>(na, nb, inbox, h_main).total;
    }
}

// One candidate plan: na weight slots, nb activation buffers, cols TMEM
// columns, at most cap bytes of shared memory. False if it does not fit.
static bool plan_fit(int npad, int cl, int t, int64_t rows, int64_t groups, int na, int nb, int cols, int cap,
                     int floor_bytes, F4Plan* out) {
    const int h_main = static_cast<int>(rows < kTileRows ? rows : kTileRows);
    const int h_tail = rows > kTileRows ? static_cast<int>(rows % kTileRows) : 0;
    const int tiles = rows <= kTileRows ? 1 : static_cast<int>(rows / kTileRows) + (h_tail ? 1 : 0);
    const int inbox = cl > 1 ? static_cast<int>(rows) * inbox_vectors(npad) * 16 : 0;
    const int sfa_col = (cols - 16 * na - 16 * nb) / 32 * 32;
    const int max_batch = sfa_col / npad;
    // A cluster hands rank 1's sums of every tile over at once, and above 8
    // tokens (128 MMA columns) x is converted only once per CTA: one batch.
    if (max_batch < 1 || ((cl > 1 || t > 8) && max_batch < tiles)) return false;
    int bytes = smem_layout_bytes(npad, na, nb, inbox, h_main) + 1024;  // + alignment slack
    if (bytes > cap) return false;
    bytes = bytes > floor_bytes ? bytes : floor_bytes;
    F4Plan r{};
    r.npad = npad;
    r.cl = cl;
    r.groups = static_cast<int>(groups);
    r.grid = static_cast<int>(groups * cl);
    r.rows = static_cast<int>(rows);
    r.h_main = h_main;
    r.h_tail = h_tail;
    r.tiles = tiles;
    r.na = na;
    r.nb = nb;
    r.max_batch = max_batch;
    r.tmem_cols = cols;
    r.inbox_bytes = inbox;
    r.smem_bytes = bytes;
    *out = r;
    return true;
}

bool plan_f4(int t, int64_t k, int64_t n, int num_sms, int max_smem, F4Plan* out, bool swiglu_in) {
    if (t < 1 || t > (swiglu_in ? 4 : 16) || k % kStageK != 0 || n < 1 || num_sms < 2) return false;
    if (k >= (int64_t(1) << 30) || n >= (int64_t(1) << 30)) return false;
    const int npad = npad_for(t);
    const int64_t stages = k / kStageK;
    // Rows per group: N over the SMs, rounded up to 8 (atoms of a tile stay
    // 1024-aligned). A lone CTA with fewer than 96 rows would feed the MMA
    // mostly missing rows; a cluster of 2 then splits K and doubles the rows.
    auto rows_for = [&](int groups) {
        const int64_t r = (n + groups - 1) / groups;
        return (r + 7) / 8 * 8;
    };
    // Up to 32 MMA columns, prefer plans two CTAs can share an SM with (at
    // most half its shared memory, 256 TMEM columns; launched with more than
    // a third of it, so never three): the next call's CTA then sets up and
    // prefetches its first weight stages while this call's CTA finishes. The
    // most weight slots (at least 3) next to 3 or 4 activation buffers
    // (kGroups stages are converted at once, and the MMA trails them). Else
    // one CTA per SM and 512 columns: up to 32 MMA columns, as many weight
    // slots as fit next to 6 (else 4) activation buffers; wider, the weight
    // ring first (its refills bound t = 8), next to 3 to 6 buffers.
    const int half = (max_smem + 1024) / 2 - 1024;
    const int third = (max_smem + 1024) / 3 + 1024;
    auto fit = [&](int cl, int64_t rows) -> bool {
        const int64_t groups = (n + rows - 1) / rows;
        if (npad <= 32 && !swiglu_in) {
            for (int na = kMaxNA; na >= 3; --na)
                for (int nb = 4; nb >= 3; --nb)
                    if (plan_fit(npad, cl, t, rows, groups, na, nb, 256, half, third, out)) return true;
            // t <= 2 with one 128-row tile per CTA (the FFN widths): 2
            // activation buffers (their conversion is short) leave room for
            // 3 weight slots within half the SM.
            if (npad == 16 && rows <= kTileRows)
                for (int na = kMaxNA; na >= 3; --na)
                    if (plan_fit(npad, cl, t, rows, groups, na, 2, 256, half, third, out)) return true;
        }
        if (npad <= 32)
            for (int nb = 6; nb >= 4; nb -= 2)
                for (int na = kMaxNA; na >= 2; --na)
                    if (plan_fit(npad, cl, t, rows, groups, na, nb, 512, max_smem, 0, out)) return true;
        for (int na = kMaxNA; na >= 2; --na)
            for (int nb = 6; nb >= 3; --nb)
                if (nb != 5 && plan_fit(npad, cl, t, rows, groups, na, nb, 512, max_smem, 0, out)) return true;
        return false;
    };
    const int64_t lone = rows_for(num_sms), pair = rows_for(num_sms / 2);
    // A cluster of 2 also when t > 4 (the conversion's cost per stage
    // doubles from t = 4 to t = 8): each rank converts half of x, and the
    // converted stage feeds twice the rows. It needs every tile of the group
    // in one batch (TMEM), else lone CTAs.
    if (stages >= 2 && (lone < 96 || npad > 32) && fit(2, pair)) return true;
    if (lone < 96 && stages >= 2) return false;
    return fit(1, lone);
}

cudaError_t launch_f4_linear(const CUtensorMap& main_map, const CUtensorMap& tail_map, const F4Params& p,
                             const F4Plan& plan, cudaStream_t stream) {
    if (p.xab) {  // t <= 4 (plan_f4)
        if (plan.npad > 32) return cudaErrorInvalidValue;
        return plan.npad == 16 ? launch_npad<16, 1>(main_map, tail_map, p, plan, stream)
                               : launch_npad<32, 1>(main_map, tail_map, p, plan, stream);
    }
    switch (plan.npad) {
        case 16: return launch_npad<16, 0>(main_map, tail_map, p, plan, stream);
        case 32: return launch_npad<32, 0>(main_map, tail_map, p, plan, stream);
        case 48: return launch_npad<48, 0>(main_map, tail_map, p, plan, stream);
        case 64: return launch_npad<64, 0>(main_map, tail_map, p, plan, stream);
        default: return launch_npad<128, 0>(main_map, tail_map, p, plan, stream);
    }
}

}  // namespace f4
}  // namespace mxfp4
