/*
 * mxfp4.h -- C ABI of the GB300 (sm_103a) MXFP4 weight-streaming library.
 *
 * The decode / speculative-verify step reads every weight it needs from HBM
 * once and applies it to the handful of tokens in the step ("Zyphra
 * Inference Wave 2", section "Speculative decoding"; AMD "megakernel-intro",
 * section "3. Low-Precision Data Types"). Weights are MXFP4: blocks of 32
 * E2M1 values (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 with a sign bit) that
 * share one E8M0 power-of-two scale, 4.25 bits per value ("Zyphra Inference
 * Wave 2", section "Quantization"). Activations are bf16 and outputs bf16
 * with fp32 accumulation (the a16w4 kernel of "Zyphra Inference Wave 2",
 * section "Kernel Results").
 *
 * Packed layout (shared by every entry point):
 *   wq  uint8 [rows, K/2]   byte j of a row holds the code of column 2j in
 *                           its low nibble and of column 2j+1 in its high
 *                           nibble; code bit 3 is the sign.
 *   ws  uint8 [rows, K/32]  E8M0 byte s of each 32-column block: 2^(s-127).
 *
 * Conventions for every call:
 *   - All pointers are device memory owned by the caller. The library
 *     allocates nothing; the MoE and FFN scratch comes from the caller's
 *     workspace. Exception: mxfp4_moe_noalloc keeps its scratch in one
 *     fixed array of the library (see there).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls
 *     only enqueue work and return; results are ready when the stream is.
 *   - Argument errors are returned before anything is launched. A failed
 *     launch returns MXFP4_ERR_CUDA.
 *   - Kernels never spin unboundedly: every wait gives up after about two
 *     seconds, sets a per-device status word and lets the kernel exit.
 *     mxfp4_last_device_status() reports (and clears) that word.
 *   - Identical inputs give bit-identical outputs (no floating-point
 *     atomics); calls are stateless and thread-safe apart from the
 *     caller's own buffers. Exception: calls of mxfp4_moe_noalloc that
 *     overlap on the GPU (unordered streams, or threads) race on its
 *     shared scratch array.
 *   - The first call on a device looks up per-device addresses (the status
 *     word, the mxfp4_moe_noalloc scratch) and keeps them for the life of
 *     the process. After cudaDeviceReset, or anything else that replaces
 *     the device's primary context, unload and reload the library.
 *   - There is no CPU path: without a GB300-class GPU every compute call
 *     returns MXFP4_ERR_CUDA.
 */
#ifndef MXFP4_H
#define MXFP4_H

#include <stddef.h>
#include <stdint.h>

/* The library is built with hidden visibility; only these declarations are
 * exported, so two builds loaded into one process never share a symbol. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MXFP4_OK = 0,
    MXFP4_ERR_INVALID_ARG = 1, /* null pointer, negative or zero size     */
    MXFP4_ERR_SHAPE = 2,       /* a size the kernels do not support       */
    MXFP4_ERR_ALIGN = 3,       /* a pointer is not aligned as documented  */
    MXFP4_ERR_WORKSPACE = 4,   /* workspace missing or too small          */
    MXFP4_ERR_CUDA = 5,        /* CUDA runtime or launch failure          */
    MXFP4_ERR_TIMEOUT = 6      /* a device-side bounded wait expired      */
} mxfp4_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* mxfp4_strerror(int status);

/*
 * MXFP4 packer ("Zyphra Inference Wave 2", section "Quantization"; the OCP
 * MX rule for the shared scale). For every 32-value block of a row:
 * amax = max |w|, s = clamp(floor(log2 amax) - 2 + 127, 0, 254) (0 for an
 * all-zero block), each value w * 2^(127-s) rounded to the nearest E2M1
 * point with ties to even and saturation at 6, keeping its sign bit.
 *   w   device float32 [n, k], row-major, 16-byte aligned, finite values
 *   n   rows (>= 1);  k  columns (>= 32, k % 32 == 0)
 *   wq  device uint8 [n, k/2], 16-byte aligned (output)
 *   ws  device uint8 [n, k/32] (output)
 * Bit-exact with the oracle. NaN/Inf inputs are not supported (their codes
 * are unspecified).
 */
int mxfp4_quantize(const float* w, int64_t n, int64_t k, uint8_t* wq, uint8_t* ws, void* stream);

/*
 * Weight-streaming linear layer, dense and LM-head shapes ("Zyphra
 * Inference Wave 2", section "Speculative decoding": one target token plus
 * drafts, or one token per concurrent request, per step):
 *   y[t][j] = bf16( sum_k x[t][k] * w[j][k] ),  w = dequantized (wq, ws)
 *   x   device bf16 [t, k], row-major, 16-byte aligned
 *   t   tokens, 1 <= t <= 32
 *   k   reduction length, k % 32 == 0, k >= 32
 *   wq  device uint8 [n, k/2], 16-byte aligned;  ws device uint8 [n, k/32],
 *       16-byte aligned
 *   n   output features (>= 1, < 2^31)
 *   y   device bf16 [t, n], row-major, 2-byte aligned (output)
 * Accumulation is fp32 (tensor-core fp32 accumulate); the summation order
 * is the kernel's. Three kernels serve the call (mxfp4_linear_plan says
 * which):
 *   - k % 512 == 0 and t <= 8, or 9 <= t <= 16 where each CTA's tiles of
 *     128 rows fit one accumulator batch (dense widths; not the LM head):
 *     the packed-E2M1 tensor-core kernel
 *     (tcgen05.mma kind::mxf4: the weight codes go from HBM to the tensor
 *     cores as stored, two per byte, with their E8M0 scales). Its other
 *     operand is E2M1 too, so each bf16 activation is written as eight
 *     E2M1 digit pieces: with E = floor(log2) of the largest magnitude of
 *     its (token, 32 values) block (at least -112), X = round(|x| 2^(15-E))
 *     has eight 2-bit digits D_p (most significant first) and
 *     x = sign * sum_p (D_p / 2) 2^(E - 2p). Exact for every value within
 *     2^8 of its block's largest magnitude; smaller ones keep an absolute
 *     error of at most 2^(E-16) (for blocks whose largest magnitude is
 *     below 2^-112, at most 2^-128: the lowest piece scale is 2^-127).
 *   - k % 512 != 0, or t >= 9 with wq not 32-byte aligned: the streaming
 *     engine (E2M1 -> f16 in registers, mma.sync, fp32 block scaling).
 *   - otherwise (9 <= t <= 32): the E4M3-split tensor-core kernel
 *     (tcgen05.mma kind::mxf8f6f4: the E2M1 codes and E8M0 scales go to
 *     the tensor cores as stored). Its other operand is 8-bit, so each bf16
 *     activation is split into two E4M3 pieces under one power-of-two scale
 *     per (token, 32 values) -- the pages' production format pairs MXFP4
 *     weights with MXFP8 activations ("Zyphra Inference Wave 2", section
 *     "Quantization"; AMD "megakernel-intro", section "3. Low-Precision
 *     Data Types"). The split is exact for values within 2^9 of their
 *     block's largest magnitude; smaller ones keep an absolute error below
 *     2^-17 of that maximum, far inside the tolerance's RSS term.
 * Returns MXFP4_ERR_SHAPE when no shared-memory plan fits. The binding
 * limit is k: a row group's scale bytes for all of k (k/2 bytes) stay on
 * chip next to the staging buffers. Every t <= 32 and n plans for
 * k <= 262144 on GB300.
 */
int mxfp4_linear(const void* x, int64_t t, int64_t k, const uint8_t* wq, const uint8_t* ws, int64_t n,
                 void* y, void* stream);

/*
 * How mxfp4_linear cuts the weight stream for one shape (the plan it would
 * launch). The pages have no counterpart to this entry point: it reports
 * the kernel's choices, which set its speed, and lets them be checked
 * without a GPU.
 *   t, k, n    as for mxfp4_linear (same argument checks)
 *   num_sms    streaming multiprocessors of the device
 *              (cudaDevAttrMultiProcessorCount; 152 on GB300)
 *   max_smem   opt-in shared memory per block in bytes
 *              (cudaDevAttrMaxSharedMemoryPerBlockOptin)
 *   out        host struct, written on MXFP4_OK (caller-owned)
 * Host only: no CUDA call, no device needed. Returns MXFP4_ERR_SHAPE when
 * mxfp4_linear would (no plan fits max_smem). It takes wq to be 32-byte
 * aligned (a mode-3 shape whose wq is not runs the streaming engine).
 */
typedef struct {
    int32_t mode;        /* 0: whole K per CTA; 1: K walked in parts per CTA;
                            2: K split over a thread-block cluster (modes 0-2:
                            the streaming engine); 3: the block-scaled
                            tensor-core kernel with E4M3 activation pieces;
                            4: the packed-E2M1 tensor-core kernel (modes 3-4:
                            cluster 2 = K split in halves) */
    int32_t ctas;        /* CTAs launched (mode 2: an upper bound; the number
                            of co-resident clusters decides) */
    int32_t cluster;     /* CTAs per cluster (1 unless mode 2) */
    int32_t stage_steps; /* K steps of 256 values per weight-ring stage */
    int32_t chunk_steps; /* K steps a consumer warp takes at a time (mode 3:
                            a whole stage) */
    int32_t ring_slots;  /* stages in the weight ring */
    int32_t part_steps;  /* mode 1: K steps per part; else 0 */
    int32_t batch_units; /* mode 1: row groups of 16 rows per batch; mode 3:
                            128-row tiles per CTA at most; mode 4: tiles of
                            at most 128 rows per group; else 0 */
    int32_t smem_bytes;  /* dynamic shared memory per CTA */
    int32_t group_rows;  /* mode 4: output rows per CTA (or per cluster), a
                            multiple of 8; else 0 */
} mxfp4_linear_plan_t;
int mxfp4_linear_plan(int64_t t, int64_t k, int64_t n, int num_sms, int max_smem, mxfp4_linear_plan_t* out);

/*
 * Bytes of device workspace mxfp4_moe needs for t tokens, e experts,
 * top_k experts per token, hidden size `hidden` and expert width `inter`.
 */
size_t mxfp4_moe_workspace_size(int64_t t, int64_t e, int top_k, int64_t hidden, int64_t inter);

/*
 * Grouped top-k mixture-of-experts layer with fused SwiGLU ("Zyphra
 * Inference Wave 2", sections "Kernel Results" and "Quantization": at low
 * concurrency a step reads only the routed experts' weights; each expert
 * receives a few token rows). For each token t:
 *   ids = the top_k largest router logits (descending, ties to the smaller
 *         expert index), g = softmax over those top_k logits;
 *   for each selected expert e: a = W1_e[0:inter] x_t (gate rows),
 *         b = W1_e[inter:2*inter] x_t (up rows), h = SiLU(a) * b (fp32),
 *         o = W2_e h;
 *   y[t] = bf16( sum over the selected experts in selection order of g*o ).
 * Only experts that some token selects have their weights read.
 *   x              device bf16 [t, hidden], 16-byte aligned
 *   t              tokens, 1 <= t <= 256
 *   hidden, inter  multiples of 32 (hidden >= 32, inter >= 32)
 *   router_logits  device float32 [t, e]
 *   e              experts, top_k <= e <= 1024;  1 <= top_k <= 16
 *   w1q, w1s       device uint8 [e, 2*inter, hidden/2], [e, 2*inter, hidden/32]
 *                  (rows 0..inter-1 gate, inter..2*inter-1 up), 16-byte aligned
 *   w2q, w2s       device uint8 [e, hidden, inter/2], [e, hidden, inter/32],
 *                  16-byte aligned
 *   y              device bf16 [t, hidden] (output)
 *   topk_ids       optional device int32 [t, top_k] output (NULL = skip)
 *   topk_w         optional device float32 [t, top_k] output (NULL = skip)
 *   workspace      device scratch of at least mxfp4_moe_workspace_size()
 *                  bytes, 256-byte aligned; its contents on entry do not
 *                  matter and are overwritten.
 * Routing indices are exact (bit-identical to the oracle); gate weights
 * are fp32.
 */
int mxfp4_moe(const void* x, int64_t t, int64_t hidden, const float* router_logits, int64_t e, int top_k,
              const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q, const uint8_t* w2s, int64_t inter,
              void* y, int32_t* topk_ids, float* topk_w, void* workspace, size_t workspace_bytes,
              void* stream);

/*
 * Bytes of device workspace mxfp4_moe_shared needs (arguments as there).
 */
size_t mxfp4_moe_shared_workspace_size(int64_t t, int64_t e, int top_k, int n_shared, int64_t hidden,
                                       int64_t inter);

/*
 * mxfp4_moe with shared experts ("Zyphra Inference Wave 2", section
 * "Quantization": a decode token uses its top-k routed experts plus the
 * layer's shared experts, e.g. 8 routed and 1 shared of 257, all MXFP4).
 * The weight arrays hold e + n_shared experts: 0..e-1 routed (selected by
 * the e router logits, exactly as in mxfp4_moe), e..e+n_shared-1 shared.
 * Every token applies every shared expert, after its routed ones, with
 * weight 1:
 *   y[t] = bf16( sum_j g_j * o_{ids_j} + sum_s o_{e+s} )   (in that order).
 * The page prints no weight for a shared expert; 1 is the plain reading.
 *   n_shared       0 <= n_shared <= 16, e + n_shared <= 1024 (0 gives
 *                  mxfp4_moe's result)
 *   w1q .. w2s     as for mxfp4_moe with e + n_shared experts
 *   topk_ids, topk_w  the routed selection only, [t, top_k]
 *   workspace      at least mxfp4_moe_shared_workspace_size() bytes
 * Every other argument, limit and error is as for mxfp4_moe.
 */
int mxfp4_moe_shared(const void* x, int64_t t, int64_t hidden, const float* router_logits, int64_t e, int top_k,
                     int n_shared, const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q, const uint8_t* w2s,
                     int64_t inter, void* y, int32_t* topk_ids, float* topk_w, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace mxfp4_ffn needs for t tokens (hidden unused).
 */
size_t mxfp4_ffn_workspace_size(int64_t t, int64_t hidden, int64_t inter);

/*
 * Dense FFN chain, up -> SwiGLU -> down (lithosai "Low-Latency Inference on
 * AMD MI355X" and AMD "megakernel-intro", section "1. Megakernels": a
 * layer's stages back to back, the next stage's weights preloaded while the
 * previous one runs). The arithmetic is one SwiGLU expert of mxfp4_moe
 * applied to every token with weight 1. For each token t:
 *   a = W1[0:inter] x_t (gate rows), b = W1[inter:2*inter] x_t (up rows),
 *   h = SiLU(a) * b (fp32), y[t] = bf16( W2 h ).
 * Two forms, chosen by shape:
 *   t <= 4 with hidden and inter multiples of 512: two launches of the
 *     packed-E2M1 tensor-core kernel on the stream. The first writes a | b
 *     in fp32 to the workspace; the second computes h = SiLU(a) * b in fp32
 *     while it converts its activations (digit pieces of h: each element
 *     within 2^(E-16) of its value, E its 32-block's largest exponent), and
 *     starts streaming W2 before the first has finished (programmatic
 *     dependent launch: it waits only where it reads a | b).
 *   otherwise: ONE persistent cooperative launch (h in the workspace),
 *     preceded by a 4-byte memset of the workspace.
 *   x              device bf16 [t, hidden], 16-byte aligned; 1 <= t <= 8
 *   hidden, inter  multiples of 32, at most 2^20 (MXFP4_ERR_SHAPE also when
 *                  the staged activations of one phase do not fit on chip)
 *   w1q, w1s       device uint8 [2*inter, hidden/2], [2*inter, hidden/32]
 *                  (gate rows first), 16-byte aligned
 *   w2q, w2s       device uint8 [hidden, inter/2], [hidden, inter/32],
 *                  16-byte aligned
 *   y              device bf16 [t, hidden] (output)
 *   workspace      device scratch of at least mxfp4_ffn_workspace_size()
 *                  bytes, 256-byte aligned; contents on entry do not matter.
 * The cooperative form's CTAs wait (bounded) for the gate/up results of all
 * the others, so the whole grid must be resident. A call that shares the
 * GPU with other work that holds SMs may therefore end in MXFP4_ERR_TIMEOUT
 * (reported as for every call) instead of a result.
 */
int mxfp4_ffn(const void* x, int64_t t, int64_t hidden, const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q,
              const uint8_t* w2s, int64_t inter, void* y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Capacity in bytes of the scratch array built into the library for
 * mxfp4_moe_noalloc (held on every GPU that loads the library).
 */
#define MXFP4_MOE_NOALLOC_SCRATCH_BYTES ((size_t)12 << 20)

/*
 * mxfp4_moe without a workspace argument, for callers that cannot allocate
 * device memory where they run the layer: plugins whose host framework's
 * memory pool owns the device memory, serving loops that forbid allocation
 * after warm-up, and latency-bound loops that cannot take cudaMalloc's
 * implicit synchronisation. The pages have no counterpart to this entry
 * point.
 *   Arguments, layouts and results are those of mxfp4_moe, minus
 *   `workspace` / `workspace_bytes`.
 *   Scratch: a fixed device array of MXFP4_MOE_NOALLOC_SCRATCH_BYTES (12 MiB)
 *   inside the library. Problems needing more (mxfp4_moe_workspace_size)
 *   return MXFP4_ERR_WORKSPACE before any launch.
 *   The first call on a device looks up the array's device address; make
 *   it before any stream capture. Calls share the array: calls that overlap
 *   on the GPU race. Nothing is allocated or freed.
 */
int mxfp4_moe_noalloc(const void* x, int64_t t, int64_t hidden, const float* router_logits, int64_t e, int top_k,
                      const uint8_t* w1q, const uint8_t* w1s, const uint8_t* w2q, const uint8_t* w2s, int64_t inter,
                      void* y, int32_t* topk_ids, float* topk_w, void* stream);

/*
 * Synchronizes `stream`, then returns MXFP4_OK, MXFP4_ERR_TIMEOUT if some
 * kernel of this library on the current device gave up a bounded wait since
 * the last call, or MXFP4_ERR_CUDA if the stream reports an error. Clears
 * the device status word.
 */
int mxfp4_last_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#endif /* MXFP4_H */
