/*
 * moe.h -- C ABI of libmoe.so: the grouped mixture-of-experts expert-FFN path
 * on one GB300 (sm_103a) GPU.
 *
 * The path has five steps, each one call below, and all of them only enqueue
 * work on the caller's CUDA stream (no host synchronisation between the
 * router and the combine, so the whole layer can be captured in a CUDA graph):
 *
 *   moe_route_topk_softmax   top-k softmax routing
 *   moe_router_topk_softmax  the router GEMM (x . Wr) in front of it
 *   moe_align_block_size     sort (token, expert) pairs into block-padded spans
 *   moe_grouped_gate_up      grouped gate/up GEMM with the SiLU-mul fused
 *   moe_grouped_down         grouped down GEMM
 *   moe_lora_grouped_down    optional per-expert LoRA shrink/expand fold
 *   moe_lora_gather_bgmv     the same fold on unsorted slot-major rows (decode)
 *   moe_combine              weighted top-k combine
 *
 * Sources the semantics are restated from (cited per call below):
 *   [lora]    spark_model/layers/ops/moe_lora_grouped.rs (Atlas inference docs)
 *   [ferrum]  ferrum-kernels 0.7.7, src/backend/cuda/moe.rs
 *   [triton]  ferrum-kernels, src/backend/cuda/triton_fused_moe.rs
 *   [cutlass] metrale_gpu_runtime/cutlass/grouped.rs
 *
 * Conventions shared by every call:
 *   - Pointers marked "device" are CUDA device addresses owned by the caller;
 *     the library never allocates, frees or retains them past the call's
 *     stream work. Scratch is passed in by the caller ("workspace").
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - Every call returns MOE_OK (0) or an error status. Misuse detectable on
 *     the host (bad sizes, NULL required pointers, misaligned addresses,
 *     limits) returns MOE_ERR_INVALID / MOE_ERR_UNSUPPORTED before anything is
 *     launched; a failed launch returns MOE_ERR_CUDA. moe_last_error() gives
 *     the calling thread's message for the last failure. Nothing aborts.
 *   - Problems only the GPU can see (an expert id out of range, inconsistent
 *     expert_offsets, a pipeline wait that gave up) are OR-ed into an optional
 *     device `err_word` (int32, caller zeroes it) as MOE_DEV_ERR_* bits; the
 *     kernels skip the offending work and return, they never trap.
 *   - A pair id is p = t * top_k + j (token t, slot j); P = T * top_k.
 *     sorted_token_ids holds pair ids, and the sentinel for a padding row is
 *     P ([triton] module doc: sentinel `total_pairs`). The token of a pair is
 *     p / top_k ([lora] gather_row_token).
 *   - bf16 / fp16 tensors are dense row-major with the last index contiguous.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------- */
#define MOE_OK 0
#define MOE_ERR_INVALID 1     /* bad argument, detected on the host, nothing launched */
#define MOE_ERR_UNSUPPORTED 2 /* valid request beyond this library's limits */
#define MOE_ERR_CUDA 3        /* a CUDA runtime call or a kernel launch failed */

/* ---- device error word bits ---------------------------------------------- */
#define MOE_DEV_ERR_EXPERT_ID 0x1 /* an expert id outside [0, E): that pair was dropped */
#define MOE_DEV_ERR_CAPACITY 0x2  /* the padded total exceeded max_padded */
#define MOE_DEV_ERR_OFFSETS 0x4   /* expert_offsets broke its invariants: no tile ran */
#define MOE_DEV_ERR_PAIR_ID 0x8   /* a sorted entry or pair row was out of range: row skipped */
#define MOE_DEV_ERR_TIMEOUT 0x10  /* a pipeline wait gave up; the kernel returned early */

/* ---- limits ---------------------------------------------------------------- */
#define MOE_MAX_EXPERTS 256 /* [ferrum] moe_align_block_size: compile-time MAX_NUM_EXPERTS */
/* Split-K area of the grouped GEMM workspaces: fp32 partial sums of up to
 * MOE_SPLITK_CTAS CTAs (128 KB each) followed by 16 bytes of flags per CTA.
 * A CTA that leaves partial sums marks them with a generation number the
 * library draws for each call (nonzero, process-wide), and the CTA that adds
 * them accepts only its own call's number, then clears the flag. So whatever
 * an earlier call left there (a call that reported a device error, or
 * uninitialised memory) is not mistaken for a finished piece. One exception:
 * a replayed CUDA graph repeats the numbers of its capture, so after a replay
 * that reported a device error, zero the area before the next replay.
 * Allocating it zeroed is recommended (a stale flag equal to a future call's
 * number is then impossible rather than unlikely). */
#define MOE_SPLITK_CTAS 256
#define MOE_SPLITK_BYTES ((size_t)MOE_SPLITK_CTAS * (131072 + 16))
#define MOE_MAX_TOPK 16
#define MOE_MAX_LORA_RANK 64

/* ---- element types ----------------------------------------------------------- */
#define MOE_ACT_BF16 0
#define MOE_ACT_F16 1

#define MOE_W_BF16 0      /* dense weight in the activation type */
#define MOE_W_GPTQ_INT4 1 /* raw GPTQ 4-bit: qweight / scales / qzeros ([triton]) */
#define MOE_W_NVFP4 2     /* E2M1 + E4M3 per-16 scales + fp32 scale2 ([cutlass]) */
#define MOE_W_FP8_E4M3 3  /* E4M3 codes + one fp32 scale per output row ([lora]: fp8 grouped weights) */

/*
 * A stacked expert weight of E experts, each of logical shape [N, K]
 * (N output features, K contraction). For the gate/up weight N = 2*I: rows
 * [0, I) are the gate projection and rows [I, 2I) the up projection. For the
 * down weight N = H and K = I. All pointers are device addresses.
 *
 *   MOE_W_BF16:  w      = [E, N, K] bf16 (the activation type must be bf16)
 *   MOE_W_GPTQ_INT4 ([triton] TritonStackedGptqWeight, raw layout, no repack):
 *                w      = qweight int32 [E, K/8, N]; nibble j (bits 4j..4j+3)
 *                         of qweight[e][i][n] is the code of k = 8i + j
 *                scales = fp16 [E, K/G, N]
 *                zeros  = qzeros int32 [E, K/G, N/8]; nibble n%8 of word n/8
 *                         is the zero point of column n, used as stored
 *                w(k, n) = (q - z) * s   (rounded to the activation type)
 *                group_size G: a multiple of 64 dividing K
 *   MOE_W_NVFP4 ([cutlass] nvfp4_grouped_gate_up: [N,K/2] and [K/16,N]):
 *                w      = packed E2M1 uint8 [E, N, K/2]; byte (n, k/2) holds
 *                         even k in its low nibble, odd k in its high nibble
 *                scales = E4M3 uint8 [E, K/16, N]
 *                scale2 = fp32 [S, E]: S = 2 for a gate/up weight (gate's E
 *                         values, then up's), S = 1 for a down weight
 *                w(n, k) = e2m1 * e4m3(scales[k/16][n]) * scale2
 *   MOE_W_FP8_E4M3 (the pages name fp8 grouped weights but print no layout;
 *                this is the plain W8A16 reading):
 *                w      = E4M3 uint8 [E, N, K] (OCP FP8: bias 7, no inf)
 *                scales = fp32 [E, N], one per output row
 *                w(n, k) = e4m3(w[n][k]) * scales[n]
 */
typedef struct MoeWeight {
    int32_t format;     /* MOE_W_* */
    int32_t group_size; /* GPTQ group size; 0 otherwise */
    const void* w;
    const void* scales;
    const void* zeros;
    const float* scale2;
} MoeWeight;

/*
 * Per-expert LoRA tables of the down-projection fold ([lora] MoeExpertRoute).
 * a_table / b_table hold one device address per expert (0 = expert
 * unadapted): A_e is bf16 [max_rank, k_in], B_e is bf16 [n_out, max_rank]
 * (max_rank is B_e's row stride), both 16-byte aligned. scale_table holds scale_e (0 where
 * unadapted). n_experts is the table length = largest adapted id + 1; experts
 * at or past it fold nothing.
 */
typedef struct MoeExpertRoute {
    const uint64_t* a_table;   /* device [n_experts] */
    const uint64_t* b_table;   /* device [n_experts] */
    const float* scale_table;  /* device [n_experts] */
    uint32_t n_experts;
    uint32_t k_in;     /* contraction of the shrink (the intermediate size) */
    uint32_t n_out;    /* output of the expand (the hidden size) */
    uint32_t max_rank; /* padded rank, <= MOE_MAX_LORA_RANK */
} MoeExpertRoute;

/* ---- library state --------------------------------------------------------- */

/* Message of the calling thread's last failed call ("" if none). The string
 * lives until the thread's next failing call. */
const char* moe_last_error(void);

/* Number of kernels this library has launched in the process so far. */
uint64_t moe_launch_count(void);

/*
 * Time limit, in nanoseconds, of every pipeline wait inside the grouped GEMM
 * kernels launched after this call (process-wide; 0 restores the default of
 * 2 s). A wait that runs out sets MOE_DEV_ERR_TIMEOUT in the call's err_word;
 * the kernel then lets its copies and MMAs in flight land, frees its tensor
 * memory and returns, so the context stays usable. (Partial sums it left in
 * a split-K area are ignored by later calls; see MOE_SPLITK_BYTES.) This is a
 * testing hook (it lets a test make the waits run out on purpose, as the
 * pages' status-return error model asks of every failure); production
 * callers leave the default. Returns the previous limit.
 */
uint64_t moe_set_wait_limit_ns(uint64_t ns);

/* ---- a1: routing --------------------------------------------------------- */

/*
 * Top-k softmax routing ([ferrum] route_topk_softmax; one warp per row).
 *   logits        device f32 [T, E]
 *   topk_ids      device i32 [T, top_k] out: experts by descending logit,
 *                 equal logits in ascending expert order
 *   topk_weights  device f32 [T, top_k] out: softmax probabilities of the
 *                 chosen experts; renormalize != 0 rescales them to sum to 1
 *                 (the page's norm_topk_prob)
 * Arithmetic (bit-exact contract): d = l - max in f32; e = f32(exp(double(d)));
 * renormalised: S = e_0 + e_1 + ... in f32 in rank order, w = e / S (IEEE
 * f32); otherwise Z sums every e_i in f32 as 32 lane partials (lane = i mod
 * 32, ascending i) followed by xor-butterfly steps 16, 8, 4, 2, 1.
 * Errors: E < 1 or E > MOE_MAX_EXPERTS, top_k < 1, top_k > E or top_k >
 * MOE_MAX_TOPK, T < 0, NULL pointers (T > 0).
 */
int moe_route_topk_softmax(const float* logits, int32_t* topk_ids, float* topk_weights,
                           int32_t T, int32_t E, int32_t top_k, int32_t renormalize,
                           void* stream);

/*
 * Router GEMM, then routing (the pages route from given logits and print no
 * router; the workloads define one):
 *     logits[t, e] = f32( sum_h x[t, h] * w_router[h, e] )
 * accumulated in f32 by fused multiply-adds in a fixed order (the same on
 * every run), then moe_route_topk_softmax on those logits (same outputs and
 * rules).
 *   x             device act [T, H], 16-byte aligned
 *   act           MOE_ACT_BF16 | MOE_ACT_F16
 *   w_router      device f32 [H, E]
 *   logits        device f32 [T, E] out (also the routing input)
 *   topk_ids / topk_weights   as moe_route_topk_softmax
 * Requirements: H % 8 == 0, 1 <= E <= MOE_MAX_EXPERTS, 1 <= top_k <= min(E,
 * MOE_MAX_TOPK).
 */
int moe_router_topk_softmax(const void* x, int32_t act, const float* w_router, int32_t T,
                            int32_t H, int32_t E, int32_t top_k, int32_t renormalize,
                            float* logits, int32_t* topk_ids, float* topk_weights, void* stream);


/* ---- a2: align ------------------------------------------------------------- */

/* Rows the sorted buffers need for P pairs: round_up(P + min(E, P) *
 * (block_size - 1), block_size). Returns -1 on bad arguments. Plays the role
 * of [ferrum]'s sorted_max_size. */
int64_t moe_align_capacity(int64_t P, int32_t E, int32_t block_size);

/* Bytes of device workspace moe_align_block_size needs for P pairs, E experts. */
size_t moe_align_workspace_size(int32_t P, int32_t E);

/*
 * Sort (token, expert) pairs by expert into spans padded to block_size
 * ([ferrum] moe_align_block_size / moe_align_block_size_pair_ids and
 * moe_build_pairs_by_token; [triton] sorted_token_ids / expert_ids contract).
 * Deterministic and stable (pairs keep ascending id order within a span).
 *   topk_ids               device i32 [P] (the router's [T, top_k], flat)
 *   sorted_token_ids       device i32 [max_padded] out: pair ids by expert,
 *                          sentinel P on padding rows and on [total, max_padded)
 *   expert_ids             device i32 [max_padded / block_size] out: the
 *                          expert of each block, -1 past the total
 *   expert_offsets         device i32 [E + 1] out: padded prefix sum, expert e
 *                          owns rows [expert_offsets[e], expert_offsets[e+1])
 *   total_tokens_post_pad  device i32 [1] out: expert_offsets[E]
 *   pair_to_row            device i32 [P] out: row of each pair, -1 if dropped
 *   err_word               device i32 [1] or NULL: MOE_DEV_ERR_EXPERT_ID
 *   workspace              device, >= moe_align_workspace_size(P, E) bytes,
 *                          16-byte aligned; contents need not be initialised
 * Errors: E < 1 or > MOE_MAX_EXPERTS, block_size < 1, P < 0, max_padded <
 * moe_align_capacity(P, E, block_size) or not a multiple of block_size,
 * workspace too small, NULL outputs.
 */
int moe_align_block_size(const int32_t* topk_ids, int32_t P, int32_t E, int32_t block_size,
                         int32_t max_padded, int32_t* sorted_token_ids, int32_t* expert_ids,
                         int32_t* expert_offsets, int32_t* total_tokens_post_pad,
                         int32_t* pair_to_row, int32_t* err_word, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * moe_align_block_size without a workspace argument, for callers that cannot
 * allocate device memory (for example an application whose framework owns
 * the whole device memory budget and gives out no allocator, or a caller that
 * must not make an allocation call, which can synchronise the device, on its
 * hot path). The source pages have no counterpart of this call.
 *
 * Same arguments, outputs and errors as moe_align_block_size, minus the
 * workspace. The scratch is a fixed array inside the library, sized for
 * P <= MOE_ALIGN_NOALLOC_MAX_PAIRS pairs and E <= MOE_MAX_EXPERTS experts
 * (about 1.1 MiB held on every GPU that loads the library until exit); a
 * larger P is rejected with MOE_ERR_INVALID. The first call on a device looks
 * up the array's device address with that device current (and so does the
 * first call after the device's context was destroyed and made again, e.g. by
 * cudaDeviceReset), so make that first call before any stream capture. Nothing is allocated or freed. All calls on
 * a device share the array: calls that overlap on the GPU (unordered streams)
 * race on it. Nothing in it needs to start at zero.
 */
#define MOE_ALIGN_NOALLOC_MAX_PAIRS 262144
int moe_align_block_size_noalloc(const int32_t* topk_ids, int32_t P, int32_t E, int32_t block_size,
                                 int32_t max_padded, int32_t* sorted_token_ids, int32_t* expert_ids,
                                 int32_t* expert_offsets, int32_t* total_tokens_post_pad,
                                 int32_t* pair_to_row, int32_t* err_word, void* stream);

/* ---- a3 / a4: grouped GEMMs ----------------------------------------------- */

/* Bytes of device workspace moe_grouped_gate_up needs: the gathered copy of
 * the activations in sorted-row order, rounded up to 256 bytes, then the
 * split-K area (MOE_SPLITK_BYTES; allocating it zeroed is recommended). */
size_t moe_gate_up_workspace_size(int32_t max_padded, int32_t H);

/*
 * Grouped gate/up GEMM with the SiLU-mul fused ([cutlass]
 * nvfp4_grouped_gate_up_fused: group row i reads token sorted_token_ids[i],
 * one grouped launch for all experts; [triton] launch_fused_moe_w4a16_triton:
 * one launch covers every (token, expert) pair, sentinel rows masked).
 * For every sorted row r of expert e holding pair p != P, t = p / top_k:
 *     h[r, n] = act( silu(x[t] . Wg_e[n]) * (x[t] . Wu_e[n]) ),  n < I,
 * with fp32 accumulation on the tensor cores and silu(g) = g / (1 + exp(-g)).
 * Padding rows are not guaranteed to be written (tiles made only of padding
 * rows are skipped); rows at or past expert_offsets[E] are not written. Tiles
 * are scheduled on the device from expert_offsets (no host sync). Batches
 * with few rows per expert (T * top_k / min(E, T * top_k) < 128) use the
 * decode form of the kernel, in which the weights are the MMA's M operand
 * and each tile covers one align block of rows.
 *   x                 device act [T, H]
 *   act               MOE_ACT_BF16 | MOE_ACT_F16
 *   w_gate_up         host pointer to a MoeWeight with N = 2*I, K = H
 *   sorted_token_ids, expert_offsets   device, from moe_align_block_size
 *   block_size        the block_size the align step padded spans to
 *   h_out             device act [max_padded, I] out
 *   err_word          device i32 or NULL
 *   workspace         device, >= moe_gate_up_workspace_size bytes, 128-byte aligned;
 *                     ends with a split-K area (see MOE_SPLITK_BYTES)
 * Requirements: H % 8 == 0, I % 8 == 0, E <= MOE_MAX_EXPERTS, all tensor
 * base addresses 16-byte aligned; GPTQ: group_size a multiple of 64 dividing
 * H and I % 32 == 0; NVFP4: H % 32 == 0 and I % 16 == 0; FP8: H % 16 == 0.
 * A contraction that is not a multiple of 64 is zero-padded on chip.
 */
int moe_grouped_gate_up(const void* x, int32_t act, const MoeWeight* w_gate_up,
                        const int32_t* sorted_token_ids, const int32_t* expert_offsets,
                        int32_t T, int32_t top_k, int32_t H, int32_t I, int32_t E,
                        int32_t block_size, int32_t max_padded, void* h_out, int32_t* err_word,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Grouped down GEMM ([cutlass] nvfp4_grouped_down: the intermediate is already
 * in expert order, no gather, writes c [M_total, N]).
 *     y[r, n] = act( h[r] . Wd_e[n] ),  n < H, for rows r of expert e.
 *   h                 device act [max_padded, I]
 *   w_down            host pointer to a MoeWeight with N = H, K = I
 *   sorted_token_ids  device, from moe_align_block_size (padding-only tiles
 *                     are skipped; T * top_k is its sentinel)
 *   block_size        the block_size the align step padded spans to
 *   y                 device act [max_padded, H] out (padding rows and rows past
 *                     expert_offsets[E] are not guaranteed to be written)
 *   workspace         device, >= moe_down_workspace_size() bytes, 128-byte
 *                     aligned: a split-K area (see MOE_SPLITK_BYTES); the
 *                     decode form cuts tiles across CTAs and adds partial sums
 *                     there
 * Requirements: I % 8 == 0, H % 8 == 0, 16-byte aligned tensors; GPTQ:
 * group_size a multiple of 64 dividing I and H % 32 == 0; NVFP4: I % 32 == 0
 * and H % 16 == 0; FP8: I % 16 == 0.
 */
int moe_grouped_down(const void* h, int32_t act, const MoeWeight* w_down,
                     const int32_t* sorted_token_ids, const int32_t* expert_offsets,
                     int32_t T, int32_t top_k, int32_t H, int32_t I, int32_t E,
                     int32_t block_size, int32_t max_padded, void* y, int32_t* err_word,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace moe_grouped_down needs (the split-K area). */
size_t moe_down_workspace_size(void);

/* ---- a5: LoRA fold ----------------------------------------------------------- */

/*
 * Device-side grouped LoRA fold over one window [row_offset, row_end) of the
 * sorted rows ([lora] moe_lora_grouped_down; argument order kept, with the
 * token count and top_k appended because sorted_token_ids holds pair ids).
 * For rows r of expert e < route->n_experts with a_table[e] != 0, inside the
 * window, holding pair p != P, whose token t = p / top_k has row_adapter[t]
 * >= 0 (or row_adapter == NULL: every row folds):
 *     xa[r - row_offset, j] = bf16( sum_i xrow[i] * A_e[j, i] )
 *     delta[n] = bf16( sum_j xa[r - row_offset, j] * B_e[n, j] )
 *     base_out[r, n] = bf16( f32(base_out[r, n]) + f32(scale_e * f32(delta[n])) )
 * (the page's base += scale * fp32(bf16(delta)); the multiply and the add are
 * separately rounded f32 operations). xrow = x[r] when x_gather == 0 (sorted
 * post-SiLU activations, the down fold) or x[t] when x_gather == 1
 * (token-major input, the gate/up fold). The sums accumulate in f32.
 *   route             host pointer; its tables are device arrays
 *   x                 device bf16 [rows, k_in] (x_gather 0) or [num_tokens, k_in]
 *   base_out          device bf16 [max_padded, n_out], folded in place
 *   expert_offsets    device i32 [>= n_experts + 1]
 *   sorted_token_ids  device i32 [>= row_end]
 *   row_adapter       device i32 [num_tokens] or NULL
 *   xa                device bf16 [>= row_end - row_offset, max_rank] scratch,
 *                     indexed by the local row r - row_offset
 * A window beyond every span folds nothing. Windows may be issued in any
 * number; one window [0, total) gives bit-identical results to any split.
 * Requirements: k_in % 8 == 0, n_out % 4 == 0, 1 <= max_rank <=
 * MOE_MAX_LORA_RANK, row_offset <= row_end.
 */
int moe_lora_grouped_down(const MoeExpertRoute* route, const void* x, void* base_out,
                          const int32_t* expert_offsets, const int32_t* sorted_token_ids,
                          const int32_t* row_adapter, void* xa, uint32_t row_offset,
                          uint32_t row_end, uint32_t x_gather, int32_t num_tokens,
                          int32_t top_k, void* stream);

/*
 * Decode-path LoRA fold on slot-major rows ([lora] moe_lora_gather_bgmv;
 * argument order kept). The rows are the flat (token, slot) pairs
 * s = t * top_k + j, s < n_slots, in that order (no expert sort). Row s folds
 * with expert e = indices[s] when e < route->n_experts, a_table[e] != 0 and
 * (row_adapter == NULL or row_adapter[s / top_k] >= 0):
 *     xa[s, j] = bf16( sum_i xrow[i] * A_e[j, i] )
 *     base_out[s, n] = bf16( f32(base_out[s, n]) + f32(scale_e * f32(bf16( sum_j xa[s, j] * B_e[n, j] ))) )
 * with xrow = x[s] (x_gather 0: slot-major rows, the down fold) or
 * x[s / top_k] (x_gather 1: token-major rows, the gate/up fold); the sums
 * accumulate in f32. Other rows of base_out and xa are left untouched.
 *   route        host pointer; its tables are device arrays
 *   x            device bf16 [n_slots, k_in] (x_gather 0) or [n_slots / top_k, k_in]
 *   base_out     device bf16 [n_slots, n_out], folded in place
 *   indices      device u32 [n_slots]: expert of each row
 *   row_adapter  device i32 [n_slots / top_k] or NULL
 *   xa           device bf16 [n_slots, max_rank] scratch
 * Requirements: k_in % 8 == 0, n_out % 4 == 0, 1 <= max_rank <=
 * MOE_MAX_LORA_RANK, top_k >= 1, x 16-byte aligned.
 */
int moe_lora_gather_bgmv(const MoeExpertRoute* route, const void* x, void* base_out,
                         const uint32_t* indices, const int32_t* row_adapter, void* xa,
                         uint32_t n_slots, uint32_t top_k, uint32_t x_gather, void* stream);

/* ---- a6: combine ------------------------------------------------------------- */

/*
 * Weighted top-k combine ([ferrum] moe_combine):
 *     out[t, n] = act( sum_{j < top_k} w[t, j] * y[pair_to_row[t*top_k + j], n] )
 * accumulated in f32 in ascending j. Pairs with pair_to_row < 0 (dropped) or
 * >= max_padded add nothing (the latter also sets MOE_DEV_ERR_PAIR_ID).
 *   y            device act [max_padded, H]
 *   pair_to_row  device i32 [T * top_k]
 *   topk_weights device f32 [T, top_k]
 *   out          device act [T, H] out
 * Requirements: H % 8 == 0, 16-byte aligned y / out.
 */
int moe_combine(const void* y, int32_t act, const int32_t* pair_to_row,
                const float* topk_weights, void* out, int32_t T, int32_t H, int32_t top_k,
                int32_t max_padded, int32_t* err_word, void* stream);

/* ---- host helper ------------------------------------------------------------- */

/*
 * Host-side check of the arrays a grouped launch reads ([cutlass]
 * ensure_group_arrays): `offsets` (host, offsets_len entries) must have
 * num_experts + 1 entries, offsets[0] >= 0 and never decrease; each of the
 * n_arrays per-expert host arrays (names[i], lens[i] entries) must have
 * exactly num_experts entries. Returns MOE_OK or MOE_ERR_INVALID with a
 * message naming the array and its length (moe_last_error()). Pure host
 * code: needs no GPU.
 */
int moe_validate_group_arrays(const char* who, int32_t num_experts, const int32_t* offsets,
                              int32_t offsets_len, const char* const* names,
                              const int32_t* lens, int32_t n_arrays);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
