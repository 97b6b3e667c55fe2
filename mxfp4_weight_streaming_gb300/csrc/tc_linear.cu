// Block-scaled tensor-core weight-streaming linear layer for sm_103a.
//
// What it computes ("Zyphra Inference Wave 2", sections "Speculative
// decoding" and "Quantization"; AMD "megakernel-intro", section "3.
// Low-Precision Data Types"):
//   y[t][n] = bf16( sum_k x[t][k] * w[n][k] ),  w = e2m1(code) * 2^(s-127)
// reading every weight byte from HBM once. The MXFP4 weights go to the
// tensor cores as they are stored: tcgen05.mma kind::mxf8f6f4 takes E2M1
// codes with one E8M0 scale per 32 values, so there is no dequantisation
// step. The other operand must be an 8-bit float with its own E8M0 block
// scales, so each bf16 activation x is split exactly into two E4M3 pieces
// under one scale 2^e per (token, 32 values):
//   x / 2^e = hi + lo,  hi = e4m3(x / 2^e),  lo = e4m3(x / 2^e - hi),
// with e = floor(log2 max|x|) - 7 (the block maximum lands in [128, 256)).
// A bf16 value has 8 significant bits; hi keeps the top 4 (rounded) and the
// remainder has at most 4, so the split is exact for every value within
// 2^9 of its block maximum; smaller values keep an absolute error below
// 2^-10 * 2^e (E4M3's subnormal step), under 2^-17 of the block maximum.
// Token t becomes the two B rows 2t (hi) and 2t+1 (lo) of one MMA, and the
// epilogue adds the two fp32 accumulator columns.
//
// Work split: a tile is 128 weight rows (the MMA's M) and a stage SA atoms
// of 128 K values. A CTA takes a contiguous range of tiles and walks K stage
// by stage over a batch of them (every batch tile's accumulator stays in
// TMEM), so each stage of activations is converted once per batch. When
// there are too few tiles to fill the GPU, a cluster of 2 CTAs shares one
// tile, each CTA taking half of K, and rank 1 hands its fp32 sums to rank 0
// through distributed shared memory (deterministic order: rank 0's K half,
// then rank 1's).
//
// One CTA per SM, warp-specialised:
//   warps 0-3  epilogue and block scales. Per (tile, stage), warp q loads
//              the E8M0 words of weight rows 32q..32q+31 (one 16-byte load
//              per row) and stores them into its quarter of TMEM as soon as
//              the MMAs that last read those columns are done (the MMA reads
//              row r's word at lane r, column base + r/32, base a multiple
//              of 4); per stage, every warp stores the
//              activation rows' words into its own quarter (each 32-row
//              quarter of the MMA reads them there); per batch, accumulators
//              (TMEM) -> registers -> hi + lo -> bf16 y (or the cluster
//              hand-off).
//   warp 4     TMA producer: per (tile, stage) one 3D copy of SA atoms x 128
//              rows of packed E2M1 (16U4_ALIGN16B: the copy unpacks 16 codes
//              per 16-byte smem chunk), L2 evict-first. One copy per stage:
//              the copy engine spends a roughly fixed time per copy, so the
//              scales are not a second copy.
//   warp 5     MMA issuer (one thread) and TMEM owner: 4 MMAs per atom of
//              128 x NPAD x 32, and tcgen05.commit to free the buffers.
//   warps 6-   converters, NG groups of W warps, one activation buffer per
//              group: per stage the hi/lo E4M3 rows (swizzled for the MMA)
//              and their scale bytes (16 per row: 4 atoms x 4 blocks).
// Every wait is bounded (device_common.cuh); on a timeout the status word
// is set and every role winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_common.cuh"
#include "tc_common.cuh"
#include "tc_linear_launch.h"

namespace mxfp4 {
namespace tc {

constexpr int kTileRows = 128;      // MMA M: weight rows per tile
constexpr int kAtomBytesA = 16384;  // one atom of the A tile in shared memory (128 rows x 128 B)
constexpr int kAtomPackedA = 8192;  // the same atom in HBM (packed codes)
constexpr int kEpilogueWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kFirstConverterWarp = 6;
constexpr int kTmemCols = 512;

// Shared-memory plan of one configuration (offsets from the 1024-aligned
// base). A buffer i: SA atoms of 128 rows x 128 B. B buffer j: NPAD rows x
// 128 B per atom (SA atoms). Then the B buffers' activation scale images,
// NPAD x 16 bytes each (row n's atom c block scales at bytes 16n + 4c ..
// 16n + 4c + 3), packed after the B buffers so that no buffer pads to 1 KB
// for them. NG converter groups of W warps, one B buffer per group.
template <int NPAD, int SA, int NA, int NG, int W>
struct Cfg {
    static constexpr int kConverters = NG * W;
    static constexpr int kThreads = (kFirstConverterWarp + kConverters) * 32;
    static constexpr int kAtomBytesB = NPAD * 128;
    static constexpr int kSlotA = SA * kAtomBytesA;
    static constexpr int kSlotB = SA * kAtomBytesB;  // a multiple of 1024 (NPAD >= 16)
    static constexpr int kImgBytes = NPAD * 16;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = NA * kSlotA;
    static constexpr int kOffImg = kOffB + NG * kSlotB;
    static constexpr int kOffBars = kOffImg + NG * kImgBytes;
    // mbarriers: fullA, emptyA, sfaReady [NA]; fullB, emptyB, sfbReady [NG];
    // accFull, accEmpty, inbox, drain; then the abort flag and the TMEM base
    // word.
    static constexpr int kNumBars = 3 * NA + 3 * NG + 4;
    static constexpr int kOffAbort = kOffBars + 8 * kNumBars;
    static constexpr int kOffTmemSlot = kOffAbort + 4;
    static constexpr int kOffInbox = (kOffTmemSlot + 4 + 127) / 128 * 128;
    // TMEM columns: batch accumulators from column 0; at the top (from a
    // multiple of 32), 16 scale columns per A buffer and per B buffer: the
    // word of atom a of the rows in quarter q at column 4a + q.
    static constexpr int kSfaCol = (kTmemCols - 16 * NA - 16 * NG) / 32 * 32;
    static constexpr int kSfbCol = kSfaCol + 16 * NA;
    static constexpr int kMaxBatch = kSfaCol / NPAD;
    static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 64, "MMA N");
    static_assert(SA == 2 || SA == 4, "stage atoms");
    // Byte of (B row n, stage atom c, 32-block kb) in a scale image.
    __device__ static uint32_t sfb_byte(int n, int c, int kb) { return static_cast<uint32_t>(n * 16 + 4 * c + kb); }
    static_assert(kSlotB % 1024 == 0, "B buffers stay 1024-aligned for the 128-byte swizzle");
    static constexpr int smem_bytes(int cl, int t) { return kOffInbox + (cl - 1) * t * kTileRows * 4; }
};

struct Bars {
    uint32_t base;
    int na, nb;
    __device__ uint32_t full_a(int s) const { return base + 8 * s; }
    __device__ uint32_t empty_a(int s) const { return base + 8 * (na + s); }
    __device__ uint32_t sfa_ready(int s) const { return base + 8 * (2 * na + s); }
    __device__ uint32_t full_b(int s) const { return base + 8 * (3 * na + s); }
    __device__ uint32_t empty_b(int s) const { return base + 8 * (3 * na + nb + s); }
    __device__ uint32_t sfb_ready(int s) const { return base + 8 * (3 * na + 2 * nb + s); }
    __device__ uint32_t acc_full() const { return base + 8 * (3 * na + 3 * nb); }
    __device__ uint32_t acc_empty() const { return base + 8 * (3 * na + 3 * nb + 1); }
    __device__ uint32_t inbox() const { return base + 8 * (3 * na + 3 * nb + 2); }
    __device__ uint32_t drain() const { return base + 8 * (3 * na + 3 * nb + 3); }
};

// The CTA's share: tiles [tile0, tile0 + ntile) in batches (sizes as even
// as possible), K stages [st0, st0 + spt) of each.
struct Work {
    int tile0, ntile;
    int nbatch;
    int st0, spt;
    uint32_t rank;
    // First tile (relative to tile0) and size of batch b.
    __device__ int batch_begin(int b) const { return ntile * b / nbatch; }
    __device__ int batch_size(int b) const { return ntile * (b + 1) / nbatch - ntile * b / nbatch; }
};

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

// ------------------------------------------------------------- producer
template <class C, int SA, int NA>
__device__ void producer(const TcLinearParams& p, const CUtensorMap* amap, const Work& w, uint32_t base,
                         const Bars& bars, const WaitCtx& wc) {
    const uint64_t policy = l2_evict_first_policy();
    asm volatile("prefetch.tensormap [%0];" ::"l"(amap) : "memory");
    Ring r;
    int issued = 0;
    bool ok = true;
    for (int b = 0; b < w.nbatch && ok; ++b) {
        const int t0 = w.tile0 + w.batch_begin(b), bt = w.batch_size(b);
        for (int k = 0; k < w.spt && ok; ++k) {
            const int atom0 = (w.st0 + k) * SA;
            for (int ti = 0; ti < bt; ++ti) {
                if (!mbar_wait(bars.empty_a(r.slot), r.phase ^ 1u, wc)) {
                    ok = false;
                    break;
                }
                const uint32_t slot = base + C::kOffA + r.slot * C::kSlotA;
                if (withhold_stage(static_cast<uint32_t>(issued))) {  // test-only builds
                    ++issued;
                    r.next(NA);
                    continue;
                }
                mbar_arrive_expect_tx(bars.full_a(r.slot), static_cast<uint32_t>(SA * kAtomPackedA));
                tma_load_3d_tc(slot, amap, 0, (t0 + ti) * kTileRows, atom0, bars.full_a(r.slot), policy);
                ++issued;
                r.next(NA);
            }
        }
    }
    if (!ok) {
        // Let the copies in flight land (bounded, whatever the abort flag
        // says) before the CTA may exit.
        int never = 0;
        const WaitCtx own{p.status, &never};
        for (int j = issued > NA ? issued - NA : 0; j < issued; ++j)
            mbar_wait(bars.full_a(j % NA), static_cast<uint32_t>((j / NA) & 1), own);
    }
}

// ----------------------------------------------------------- MMA issuer
// One thread issues everything, so its own instruction count sets the MMA
// rate: descriptors are per-buffer bases computed once, plus compile-time
// offsets (the start-address field of a descriptor is the byte address / 16
// in its low bits, so an offset inside a buffer is a plain add).
template <class C, int NPAD, int SA, int NA, int NG>
__device__ bool mma_issue_all(const Work& w, uint32_t base, uint32_t tbase, const Bars& bars, const WaitCtx& wc) {
    uint64_t adesc[NA], bdesc[NG];
#pragma unroll
    for (int s = 0; s < NA; ++s) adesc[s] = operand_desc(base + C::kOffA + s * C::kSlotA);
#pragma unroll
    for (int s = 0; s < NG; ++s) bdesc[s] = operand_desc(base + C::kOffB + s * C::kSlotB);
    Ring ra, rb;
    for (int b = 0; b < w.nbatch; ++b) {
        const int bt = w.batch_size(b);
        if (!mbar_wait(bars.acc_empty(), (static_cast<uint32_t>(b) & 1u) ^ 1u, wc)) return false;
        for (int k = 0; k < w.spt; ++k) {
            const int off = ((w.st0 + k) * SA) & 3;  // the stage's first atom within its 4-atom scale group
            uint64_t bd = 0;
#pragma unroll
            for (int s = 0; s < NG; ++s)
                if (s == rb.slot) bd = bdesc[s];
            const uint32_t sfb = tbase + C::kSfbCol + rb.slot * 16;
            for (int ti = 0; ti < bt; ++ti) {
                // The stage's activations and their scales (first tile only),
                // the tile's weights and its scales: all tested at once, and
                // waited for one by one (bounded) only if some are not there.
                const bool ready =
                    ti == 0 ? mbar_test4(bars.full_b(rb.slot), rb.phase, bars.sfb_ready(rb.slot), rb.phase,
                                         bars.full_a(ra.slot), ra.phase, bars.sfa_ready(ra.slot), ra.phase)
                            : mbar_test2(bars.full_a(ra.slot), ra.phase, bars.sfa_ready(ra.slot), ra.phase);
                if (!ready) {
                    if (ti == 0 && !mbar_wait(bars.full_b(rb.slot), rb.phase, wc)) return false;
                    if (ti == 0 && !mbar_wait(bars.sfb_ready(rb.slot), rb.phase, wc)) return false;
                    if (!mbar_wait(bars.full_a(ra.slot), ra.phase, wc)) return false;
                    if (!mbar_wait(bars.sfa_ready(ra.slot), ra.phase, wc)) return false;
                }
                fence_after_sync();
                uint64_t ad = 0;
#pragma unroll
                for (int s = 0; s < NA; ++s)
                    if (s == ra.slot) ad = adesc[s];
                const uint32_t sfa = tbase + C::kSfaCol + ra.slot * 16 + 4 * off;
                const uint32_t d_tmem = tbase + ti * NPAD;
                const bool acc0 = k != 0;
#pragma unroll
                for (int c = 0; c < SA; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mxf8f6f4(d_tmem, ad + static_cast<uint64_t>((c * kAtomBytesA + 32 * kk) >> 4),
                                     bd + static_cast<uint64_t>((c * C::kAtomBytesB + 32 * kk) >> 4),
                                     mma_idesc(kFmtE2M1, kFmtE4M3, kTileRows, NPAD, kk), sfa + 4 * c, sfb + 4 * c,
                                     (c | kk) != 0 || acc0);
                commit_to(bars.empty_a(ra.slot));
                ra.next(NA);
            }
            commit_to(bars.empty_b(rb.slot));
            rb.next(NG);
        }
        commit_to(bars.acc_full());
    }
    return true;
}

template <class C, int NPAD, int SA, int NA, int NG>
__device__ void mma_issuer(const Work& w, uint32_t base, uint32_t tbase, const Bars& bars, const WaitCtx& wc) {
    if (mma_issue_all<C, NPAD, SA, NA, NG>(w, base, tbase, bars, wc)) return;
    // Aborted: MMAs issued so far may still read shared memory and write
    // TMEM. One more commit tracks them all; wait for it (bounded, whatever
    // the abort flag says) before the CTA frees TMEM and exits.
    commit_to(bars.drain());
    int never = 0;
    const WaitCtx own{wc.status, &never};
    mbar_wait(bars.drain(), 0, own);
}

// ------------------------------------------------------------ converter
// One 32-value block of token t: hi/lo E4M3 bytes (32 each) and the block's
// E8M0 scale byte.
__device__ __forceinline__ void split_block(const uint4 (&v)[4], uint32_t (&hi)[8], uint32_t (&lo)[8],
                                            uint32_t& sbyte) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(v);
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) m = __vmaxu2(m, w[j] & 0x7fff7fffu);
    const uint32_t amax = max(m & 0xffffu, m >> 16);
    // e = floor(log2 amax) - 7, kept inside E8M0's range [-127, 127]; the
    // bf16 exponent field gives floor(log2) exactly (subnormals: the top
    // mantissa bit).
    int fl;
    const uint32_t ex = amax >> 7;
    if (ex != 0)
        fl = static_cast<int>(ex) - 127;
    else if (amax != 0)
        fl = (31 - __clz(static_cast<int>(amax))) - 133;
    else
        fl = 7 - 127;  // all zero: any scale; every piece is 0
    const int e = max(fl - 7, -127);
    sbyte = static_cast<uint32_t>(e + 127);
    const float f = __int_as_float((127 - e) << 23);  // 2^-e, e in [-127, 120]: a normal float
    const uint64_t f2 = f32x2_pack(f, f);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float2 s = f32x2_unpack(
            f32x2_mul(f32x2_pack(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u)), f2));
        // x / 2^e is exact in f16 for every value the E4M3 pieces can hold
        // (|v| < 256; values below 2^-17 round to zero either way).
        const __half2 h = __floats2half2_rn(s.x, s.y);
        __half2_raw hr = h;
        const __nv_fp8x2_storage_t h8 = __nv_cvt_halfraw2_to_fp8x2(hr, __NV_SATFINITE, __NV_E4M3);
        const __half2 hb = __half2(__nv_cvt_fp8x2_to_halfraw2(h8, __NV_E4M3));
        const __half2 r = __hsub2(h, hb);  // exact: the remainder of a 4-bit rounding
        __half2_raw rr = r;
        const __nv_fp8x2_storage_t l8 = __nv_cvt_halfraw2_to_fp8x2(rr, __NV_SATFINITE, __NV_E4M3);
        if (j & 1) {
            hi[j >> 1] |= static_cast<uint32_t>(h8) << 16;
            lo[j >> 1] |= static_cast<uint32_t>(l8) << 16;
        } else {
            hi[j >> 1] = h8;
            lo[j >> 1] = l8;
        }
    }
}

// Byte address of 16-byte chunk `chunk` (0-7) of row `row` of an atom in
// the 128-byte-swizzled K-major layout.
__device__ __forceinline__ uint32_t swz(uint32_t atom_base, int row, int chunk) {
    return atom_base + (row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4);
}

// Activation blocks of one stage held by a lane: block (lane + 32 u) of the
// stage's T * 4 * SA blocks (token-major), for u < kBlocksPerLane.
template <int kBlocksPerLane>
struct XBlocks {
    uint4 v[kBlocksPerLane][4];
};

template <int SA, int G>
__device__ __forceinline__ void load_blocks(const TcLinearParams& p, int atom0, int b0, int lane, XBlocks<G>& xb) {
    constexpr int kBlocksPerToken = 4 * SA;
    const int nblocks = p.T * kBlocksPerToken;
    const __nv_bfloat16* xs = p.x + static_cast<size_t>(atom0) * 128;
#pragma unroll
    for (int u = 0; u < G; ++u) {
        const int blk = b0 + lane + 32 * u;
        if (blk < nblocks) {
            const int t = blk / kBlocksPerToken, b = blk % kBlocksPerToken;
            // Through L2 only: x may have been written by the previous kernel
            // of the stream, which this kernel overlaps.
            const uint4* src = reinterpret_cast<const uint4*>(xs + static_cast<size_t>(t) * p.K + b * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) xb.v[u][q] = __ldcg(src + q);
        }
    }
}

template <class C, int SA, int G>
__device__ __forceinline__ void convert_blocks(const TcLinearParams& p, int b0, int lane, const XBlocks<G>& xb,
                                               uint32_t b_smem, uint32_t img) {
    constexpr int kBlocksPerToken = 4 * SA;
    const int nblocks = p.T * kBlocksPerToken;
#pragma unroll
    for (int u = 0; u < G; ++u) {
        const int blk = b0 + lane + 32 * u;
        if (blk >= nblocks) break;
        const int t = blk / kBlocksPerToken, b = blk % kBlocksPerToken;
        const int c = b >> 2, kb = b & 3;
        uint32_t hi[8], lo[8], sbyte;
        split_block(xb.v[u], hi, lo, sbyte);
        const uint32_t atom = b_smem + c * C::kAtomBytesB;
        const int rh = 2 * t, rl = 2 * t + 1;
        sts128(swz(atom, rh, 2 * kb), hi[0], hi[1], hi[2], hi[3]);
        sts128(swz(atom, rh, 2 * kb + 1), hi[4], hi[5], hi[6], hi[7]);
        sts128(swz(atom, rl, 2 * kb), lo[0], lo[1], lo[2], lo[3]);
        sts128(swz(atom, rl, 2 * kb + 1), lo[4], lo[5], lo[6], lo[7]);
        const uint32_t a_h = img + C::sfb_byte(rh, c, kb);
        const uint32_t a_l = img + C::sfb_byte(rl, c, kb);
        asm volatile("st.shared.u8 [%0], %1;" ::"r"(a_h), "r"(sbyte) : "memory");
        asm volatile("st.shared.u8 [%0], %1;" ::"r"(a_l), "r"(sbyte) : "memory");
    }
}

// Converter warp cw: member m of group g (W warps per group). Group g
// fills B buffer g with chunks g, g + NG, ...; member m converts blocks
// lane + 32 * (m + W * u) of each chunk.
template <class C, int NPAD, int SA, int NG, int W>
__device__ void converter(const TcLinearParams& p, int cw, int lane, const Work& w, uint32_t base, const Bars& bars,
                          const WaitCtx& wc) {
    pdl_wait_previous();  // x may come from the previous kernel of the stream
    constexpr int G = 4;  // blocks per lane in flight
    const int g = cw / W, m = cw % W;
    const int nchunks = w.nbatch * w.spt;
    const uint32_t b_smem = base + C::kOffB + g * C::kSlotB;
    const uint32_t img = base + C::kOffImg + g * C::kImgBytes;
    const int nblocks = p.T * 4 * SA;
    for (int i = g, r = 0; i < nchunks; i += NG, ++r) {
        const int atom0 = (w.st0 + i % w.spt) * SA;
        // The first group's loads go out before the buffer is free.
        XBlocks<G> xb;
        load_blocks<SA, G>(p, atom0, 32 * m * G, lane, xb);
        if (!__all_sync(0xffffffffu, mbar_wait(bars.empty_b(g), (static_cast<uint32_t>(r) & 1u) ^ 1u, wc))) return;
        convert_blocks<C, SA, G>(p, 32 * m * G, lane, xb, b_smem, img);
        for (int b0 = 32 * G * (m + W); b0 < nblocks; b0 += 32 * G * W) {
            load_blocks<SA, G>(p, atom0, b0, lane, xb);
            convert_blocks<C, SA, G>(p, b0, lane, xb, b_smem, img);
        }
        fence_proxy_async_shared();  // generic-proxy writes -> visible to the tensor core's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.full_b(g));
    }
}

// ------------------------------------------------------------- epilogue
// The 16-column TMEM scale group of one buffer, written by warp q into its
// own 32 lanes: word a (atom a of the 4-atom group) at column 4a + q.
__device__ __forceinline__ void store_scale_words(uint32_t taddr, int q, const uint4& v) {
    uint32_t c16[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) c16[i] = 0u;
    switch (q) {  // warp-uniform
        case 0: c16[0] = v.x; c16[4] = v.y; c16[8] = v.z; c16[12] = v.w; break;
        case 1: c16[1] = v.x; c16[5] = v.y; c16[9] = v.z; c16[13] = v.w; break;
        case 2: c16[2] = v.x; c16[6] = v.y; c16[10] = v.z; c16[14] = v.w; break;
        default: c16[3] = v.x; c16[7] = v.y; c16[11] = v.z; c16[15] = v.w; break;
    }
    tmem_store16(taddr, c16);
    tmem_wait_st();
    fence_before_sync();
}

// Activation scale words into one warp's 32 lanes. Each 32-row quarter of
// the MMA reads the B scales from its own lanes: B row n at lane n % 32 of
// the quarter, column (scale address + n/32). So every warp stores word a
// of B rows l (v0) and l + 32 (v1) at columns 4a and 4a + 1.
__device__ __forceinline__ void store_b_scale_words(uint32_t taddr, const uint4& v0, const uint4& v1) {
    const uint32_t c16[16] = {v0.x, v1.x, 0u, 0u, v0.y, v1.y, 0u, 0u, v0.z, v1.z, 0u, 0u, v0.w, v1.w, 0u, 0u};
    tmem_store16(taddr, c16);
    tmem_wait_st();
    fence_before_sync();
}

// Warp q of the epilogue group. Per stage it stores the activation scale
// words into its quarter; per (tile, stage) the weight scale words of rows
// 32q..32q+31; per batch it turns the accumulators into y.
template <class C, int NPAD, int SA, int NA, int NG>
__device__ void epilogue(const TcLinearParams& p, int q, int lane, const Work& w, uint32_t base, uint32_t tbase,
                         const Bars& bars, const WaitCtx& wc) {
    const int T = p.T;
    const uint32_t inbox = base + C::kOffInbox;
    bool waited = false;  // for the previous kernel of the stream (before the first write of y)
    const int rt = q * 32 + lane;  // row within a tile
    const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
    Ring ra, rb;
    for (int b = 0; b < w.nbatch; ++b) {
        const int bt = w.batch_size(b), tb = w.tile0 + w.batch_begin(b);
        // Scales of every (stage, tile) of the batch, in streaming order. The
        // MMA starts each stage with its activation scales, so those go
        // before the stage's weight scales - except for the batch's first
        // min(NA, bt) items, whose TMEM slots were freed by MMAs of earlier
        // batches: they are stored first, while x is still being produced.
        const int pre = min(NA, bt);
        for (int k = 0; k < w.spt; ++k) {
            const int group = ((w.st0 + k) * SA) >> 2;  // 4-atom scale group of the stage
            auto weight_scales = [&](int ti) -> bool {
                // The row's 16 scale bytes of the group (weights do not come
                // from the previous kernel, so the read-only path is fine).
                const int row = (tb + ti) * kTileRows + rt;
                const uint4 v = row < p.N ? __ldg(reinterpret_cast<const uint4*>(p.ws + static_cast<size_t>(row) *
                                                                                    p.nblk) + group)
                                          : make_uint4(0u, 0u, 0u, 0u);
                // The buffer's TMEM columns are free once the MMAs of the
                // stage NA items back have completed (their commit).
                if (!__all_sync(0xffffffffu, mbar_wait(bars.empty_a(ra.slot), ra.phase ^ 1u, wc))) return false;
                fence_after_sync();
                store_scale_words(tbase + lanes + C::kSfaCol + ra.slot * 16, q, v);
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.sfa_ready(ra.slot));
                ra.next(NA);
                return true;
            };
            if (k == 0)
                for (int ti = 0; ti < pre; ++ti)
                    if (!weight_scales(ti)) return;
            if (!__all_sync(0xffffffffu, mbar_wait(bars.full_b(rb.slot), rb.phase, wc))) return;
            {
                const uint32_t img = base + C::kOffImg + rb.slot * C::kImgBytes;
                const uint4 v0 = lds128(img + lane * 16);
                const uint4 v1 = NPAD > 32 ? lds128(img + (lane + 32) * 16) : make_uint4(0u, 0u, 0u, 0u);
                store_b_scale_words(tbase + lanes + C::kSfbCol + rb.slot * 16, v0, v1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.sfb_ready(rb.slot));
            rb.next(NG);
            for (int ti = (k == 0 ? pre : 0); ti < bt; ++ti)
                if (!weight_scales(ti)) return;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bars.acc_full(), static_cast<uint32_t>(b) & 1u, wc))) return;
        fence_after_sync();
        if (!waited) {
            pdl_wait_previous();  // the previous kernel may still read y
            waited = true;
        }
        for (int ti = 0; ti < bt; ++ti) {
            uint32_t r[NPAD];
            tmem_load<NPAD>(tbase + lanes + ti * NPAD, r);
            tmem_wait_ld();
            float s[NPAD / 2];
#pragma unroll
            for (int t = 0; t < NPAD / 2; ++t) s[t] = __uint_as_float(r[2 * t]) + __uint_as_float(r[2 * t + 1]);
            const int row = (tb + ti) * kTileRows + rt;
            if (p.cl > 1) {
                if (w.rank != 0) {
                    // Hand the fp32 sums to rank 0's inbox, slot rank - 1.
                    const uint32_t dst = map_to_rank(inbox, 0) + ((w.rank - 1) * T * kTileRows + rt) * 4;
#pragma unroll
                    for (int t = 0; t < NPAD / 2; ++t)
                        if (t < T) st_cluster_f32(dst + t * kTileRows * 4, s[t]);
                    fence_acq_rel_cluster();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_remote(map_to_rank(bars.inbox(), 0));
                    continue;
                }
                if (!__all_sync(0xffffffffu, mbar_wait(bars.inbox(), 0, wc))) return;
                fence_acq_rel_cluster();
                for (int rr = 1; rr < p.cl; ++rr) {
#pragma unroll
                    for (int t = 0; t < NPAD / 2; ++t)
                        if (t < T)
                            s[t] += __uint_as_float(
                                lds_u32_volatile(inbox + (((rr - 1) * T + t) * kTileRows + rt) * 4));
                }
            }
            if (row < p.N) {
#pragma unroll
                for (int t = 0; t < NPAD / 2; ++t)
                    if (t < T) p.y[static_cast<size_t>(t) * p.N + row] = __float2bfloat16_rn(s[t]);
            }
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.acc_empty());
    }
}

// --------------------------------------------------------------- kernel
template <int NPAD, int SA, int NA, int NG, int W>
__global__ void __launch_bounds__(Cfg<NPAD, SA, NA, NG, W>::kThreads, 1)
    tc_linear_kernel(const __grid_constant__ CUtensorMap amap, const TcLinearParams p) {
    using C = Cfg<NPAD, SA, NA, NG, W>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();

    Work w;
    w.rank = p.cl > 1 ? cluster_ctarank() : 0u;
    const int group = p.cl > 1 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int ngroups = p.cl > 1 ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);
    w.tile0 = static_cast<int>(static_cast<int64_t>(p.tiles) * group / ngroups);
    w.ntile = static_cast<int>(static_cast<int64_t>(p.tiles) * (group + 1) / ngroups) - w.tile0;
    w.nbatch = (w.ntile + C::kMaxBatch - 1) / C::kMaxBatch;
    w.st0 = p.stages * static_cast<int>(w.rank) / p.cl;
    w.spt = p.stages * (static_cast<int>(w.rank) + 1) / p.cl - w.st0;

    const Bars bars{base + C::kOffBars, NA, NG};
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffAbort);
    const WaitCtx wc{p.status, abort_flag};
    const uint32_t tslot = base + C::kOffTmemSlot;

    if (warp == kMmaWarp) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        for (int s = 0; s < NA; ++s) {
            mbar_init(bars.full_a(s), 1);
            mbar_init(bars.empty_a(s), 1);
            mbar_init(bars.sfa_ready(s), kEpilogueWarps);
        }
        for (int s = 0; s < NG; ++s) {
            mbar_init(bars.full_b(s), W);
            mbar_init(bars.empty_b(s), 1);
            mbar_init(bars.sfb_ready(s), kEpilogueWarps);
        }
        mbar_init(bars.acc_full(), 1);
        mbar_init(bars.acc_empty(), kEpilogueWarps);
        mbar_init(bars.inbox(), static_cast<uint32_t>((p.cl > 1 ? p.cl - 1 : 1) * kEpilogueWarps));
        mbar_init(bars.drain(), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    // B buffers start at zero: padding rows (tokens beyond T) and unused
    // scale-image bytes stay zero for the whole kernel.
    for (int i = threadIdx.x; i < (C::kOffBars - C::kOffB) / 16; i += C::kThreads)  // buffers and images
        sts128(base + C::kOffB + 16 * i, 0u, 0u, 0u, 0u);
    fence_proxy_async_shared();
    fence_before_sync();
    if (p.cl > 1)
        cluster_sync_all();
    else
        __syncthreads();
    fence_after_sync();
    const uint32_t tbase = lds_u32_volatile(tslot);

    if (w.ntile > 0 && w.spt > 0) {
        if (warp == kProducerWarp) {
            if (lane == 0) producer<C, SA, NA>(p, &amap, w, base, bars, wc);
        } else if (warp == kMmaWarp) {
            if (lane == 0) mma_issuer<C, NPAD, SA, NA, NG>(w, base, tbase, bars, wc);
        } else if (warp >= kFirstConverterWarp) {
            converter<C, NPAD, SA, NG, W>(p, warp - kFirstConverterWarp, lane, w, base, bars, wc);
        } else {
            epilogue<C, NPAD, SA, NA, NG>(p, warp, lane, w, base, tbase, bars, wc);
        }
    }
    __syncwarp();
    fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        fence_after_sync();
        tmem_dealloc(tbase, kTmemCols);
    }
    // No CTA of a cluster leaves while a peer may still write to it.
    if (p.cl > 1) cluster_sync_all();
}

// ----------------------------------------------------------------- host
template <int NPAD, int SA, int NA, int NG, int W>
struct Launcher {
    using C = Cfg<NPAD, SA, NA, NG, W>;
    static constexpr int kSA = SA;
    static constexpr int kNA = NA;
    static int smem(int cl, int t) { return C::smem_bytes(cl, t) + 1024; }
    static cudaError_t launch(const CUtensorMap& amap, const TcLinearParams& p, int grid, cudaStream_t stream) {
        static int configured[64] = {0};
        const int bytes = smem(p.cl, p.T);
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 0 || dev >= 64 || configured[dev] < bytes) {
            cudaError_t e = cudaFuncSetAttribute(tc_linear_kernel<NPAD, SA, NA, NG, W>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) configured[dev] = bytes;
        }
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[2];
        cfg.blockDim = dim3(C::kThreads);
        cfg.gridDim = dim3(grid);
        cfg.dynamicSmemBytes = bytes;
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
        cudaError_t e = cudaLaunchKernelEx(&cfg, tc_linear_kernel<NPAD, SA, NA, NG, W>, amap, p);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
};

// Configurations (NPAD, SA, NA, NG, W) by token count. Lone CTAs take
// 4-atom stages wherever the activation buffers leave room for three of them
// (a copy of 4 atoms costs the copy engine about as long as one of 2, so
// stages of 4 halve that cost per byte); T > 16 fits only 2-atom stages. A
// cluster of 2 that splits K needs T x 128 x 4 more bytes for its inbox,
// so the split configurations keep smaller rings.
using CfgT8 = Launcher<16, 4, 3, 3, 1>;        // lone and split
using CfgT16 = Launcher<32, 4, 3, 2, 2>;       // lone
using CfgT16Split = Launcher<32, 2, 5, 3, 1>;  // split
using CfgT32 = Launcher<64, 2, 5, 3, 2>;       // lone
using CfgT32Split = Launcher<64, 2, 4, 3, 2>;  // split

// Token counts below this go to the streaming engine, which measured faster
// there on GB300: its weight ring holds packed codes (one smem byte per HBM
// byte, against two for the unpacked E2M1 operand here), so a call's whole
// weight share per SM is already on chip when the previous call ends, and
// at t <= 4 its CUDA-core staging and mma.sync work keep up. From t = 5 the
// tensor-core kernel is faster (at t = 16 and 32 by 1.3x and 2.3x).
constexpr int kMinTokens = 5;

enum CfgId { kT8, kT16, kT16Split, kT32, kT32Split };

static CfgId cfg_id(int t, int cl) {
    if (t <= 8) return kT8;
    if (t <= 16) return cl > 1 ? kT16Split : kT16;
    return cl > 1 ? kT32Split : kT32;
}

static int cfg_atoms(CfgId id) {
    switch (id) {
        case kT8: return CfgT8::kSA;
        case kT16: return CfgT16::kSA;
        case kT16Split: return CfgT16Split::kSA;
        case kT32: return CfgT32::kSA;
        default: return CfgT32Split::kSA;
    }
}

static int cfg_slots(CfgId id) {
    switch (id) {
        case kT8: return CfgT8::kNA;
        case kT16: return CfgT16::kNA;
        case kT16Split: return CfgT16Split::kNA;
        case kT32: return CfgT32::kNA;
        default: return CfgT32Split::kNA;
    }
}

static int cfg_smem(CfgId id, int cl, int t) {
    switch (id) {
        case kT8: return CfgT8::smem(cl, t);
        case kT16: return CfgT16::smem(cl, t);
        case kT16Split: return CfgT16Split::smem(cl, t);
        case kT32: return CfgT32::smem(cl, t);
        default: return CfgT32Split::smem(cl, t);
    }
}

int atoms_per_stage(int t, int cl) { return cfg_atoms(cfg_id(t, cl)); }

bool plan_tc(int t, int64_t k, int64_t n, int num_sms, int max_smem, TcPlan* out) {
    // k % 512: every stage lies inside one 4-atom scale group, whose 16
    // bytes per row are one aligned vector load.
    if (t < kMinTokens || t > 32 || k % 512 != 0 || n < 1) return false;
    const int64_t tiles = (n + kTileRows - 1) / kTileRows;
    if (k / 128 >= (int64_t(1) << 30) || tiles >= (int64_t(1) << 30)) return false;
    // A cluster of 2 splits K when one tile per CTA would leave half the
    // SMs idle (one tile per cluster; every CTA keeps >= 1 stage).
    int cl = 1;
    if (2 * tiles <= num_sms) {
        const CfgId s2 = cfg_id(t, 2);
        if (k / 128 / cfg_atoms(s2) >= 2 && cfg_smem(s2, 2, t) <= max_smem) cl = 2;
    }
    const CfgId id = cfg_id(t, cl);
    if (cfg_smem(id, cl, t) > max_smem) return false;
    TcPlan r{};
    r.cl = cl;
    r.grid = cl > 1 ? static_cast<int>(cl * tiles) : static_cast<int>(tiles < num_sms ? tiles : num_sms);
    r.atoms_per_stage = cfg_atoms(id);
    r.stages = static_cast<int>(k / 128 / r.atoms_per_stage);
    r.tiles = static_cast<int>(tiles);
    r.ring_slots = cfg_slots(id);
    r.smem_bytes = cfg_smem(id, cl, t);
    *out = r;
    return true;
}

cudaError_t launch_tc_linear(const CUtensorMap& amap, const TcLinearParams& p, const TcPlan& plan,
                             cudaStream_t stream) {
    switch (cfg_id(p.T, plan.cl)) {
        case kT8: return CfgT8::launch(amap, p, plan.grid, stream);
        case kT16: return CfgT16::launch(amap, p, plan.grid, stream);
        case kT16Split: return CfgT16Split::launch(amap, p, plan.grid, stream);
        case kT32: return CfgT32::launch(amap, p, plan.grid, stream);
        default: return CfgT32Split::launch(amap, p, plan.grid, stream);
    }
}

}  // namespace tc
}  // namespace mxfp4
