/*
 * dg.h -- C ABI of the GB300 (sm_103a) block-diffusion denoising-step library
 * (libdg.so).  One denoising step of DiffusionGemma-style block diffusion over
 * a 256-token canvas: bidirectional canvas attention, the LM head with a fused
 * entropy / Gumbel-max / argmax epilogue, entropy-bounded acceptance with
 * uniform renoise, and the adaptive stop test; plus the block loop around it.
 *
 * Sources, by page title and section:
 *   "DiffusionGemma Lab", section 2 "The generation algorithm, as written in
 *     the code", items 1-7 (uniform canvas init, the acceptance rule
 *     cumsum(H) - max(H) <= 0.1, the stop rule, the 0.8 -> 0.4 temperature
 *     schedule, the argmax output, shared encoder/decoder weights, the full
 *     256-token canvas).
 *   "DiffusionGemma: Parallel Denoising From an Autoregressive Checkpoint",
 *     section "Finding" (causal encoder KV cache + bidirectional canvas
 *     decoder; the three sampler bullets; the H100 cost breakdown that names
 *     full-vocabulary softmax and canvas attention as per-step costs).
 *
 * Conventions (all entry points):
 *   - Every pointer argument is caller-owned memory.  Tensor arguments are
 *     DEVICE pointers unless the name says host.  bf16 tensors are passed as
 *     uint16_t bit patterns.  All tensors are dense row-major (last dimension
 *     contiguous) and 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy stream).
 *     Calls are asynchronous on that stream.  No call allocates device memory
 *     in the hot path: scratch comes from the caller's workspace, sized by the
 *     matching *_workspace() query (which touches no GPU).  A workspace is
 *     zero-filled by the caller before its first use, and again after a
 *     device-side error was reported in it; between calls the library leaves
 *     it in a state the next call expects.  Calls that share a workspace are
 *     ordered on one stream.
 *   - Return value: a dg_status.  It reports host-side validation (checked
 *     before anything is launched) and launch errors.  Kernels that detect a
 *     problem on the device (a bounded wait that ran out, a bounds check)
 *     record it in the status word at the start of the workspace and return
 *     early; read it with dg_read_device_status().
 *   - Supported shapes are listed per call; anything else returns
 *     DG_ERR_UNSUPPORTED without launching.
 *   - Kernel choice: the library picks the LM-head and attention kernels and
 *     their tilings from the shapes and the SM count (dg_lm_head_plan reports
 *     the LM-head choice, dg_canvas_step_plan the whole step's, for any SM
 *     count).  For testing and tuning, the environment variables
 *     DG_LM_KERNEL (single | duo | fused), DG_LM_BN (tile width),
 *     DG_LM_EPI (8 | 16: epilogue warps of the 2-SM kernel, bf16 operands),
 *     DG_ATTN_KERNEL (single | pair), DG_ATTN_SPLITS (key splits) and
 *     DG_ATTN_RESERVE (SMs kept for the attention in dg_canvas_step) force a
 *     choice; a choice the shapes do not allow is ignored.  Results do not
 *     depend on the choice beyond floating-point summation order.
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dg_status {
    DG_OK = 0,
    DG_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad value   */
    DG_ERR_UNSUPPORTED = 2,   /* shape outside the supported set              */
    DG_ERR_ALIGNMENT = 3,     /* a tensor pointer is not 16-byte aligned      */
    DG_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required   */
    DG_ERR_CUDA = 5,          /* a CUDA runtime call failed                   */
    DG_ERR_TIMEOUT = 6,       /* device: a bounded wait ran out               */
    DG_ERR_DEVICE = 7         /* device: a bounds/consistency check failed    */
} dg_status;

/* Static, never-NULL description of a status code. */
const char *dg_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int dg_version(void);

/* Device-side checks, off by default (a debugging aid; the pages describe   */
/* no failure handling).  When on, the combine / acceptance kernels check    */
/* every sampled and argmax index against [0, V), every entropy and the      */
/* canvas total for finiteness and every rank of the acceptance's ordered    */
/* positions against their count; the attention                               */
/* kernels and the split merge check each row's softmax sum and outputs for  */
/* finiteness; the MoE routing checks expert ids, positions and the token    */
/* count.  A failed check records DG_ERR_DEVICE (and a location code) in the */
/* call's workspace status word, read with dg_read_device_status (or        */
/* dg_noalloc_read_device_status), and an out-of-range index is replaced by  */
/* 0 before it is stored; results are otherwise those of the unchecked       */
/* kernels.  The setting is process-wide, read when a call enqueues its      */
/* kernels (a graph the caller captures keeps the setting of its capture;   */
/* dg_generate_block keeps one graph per setting).  Returns DG_OK.          */
int dg_set_device_checks(int on);
int dg_device_checks(void);

/* Device status word kept in the first bytes of every workspace: 0 when no
 * kernel has reported a problem, else a DG_ERR_* code.  Reads it with a
 * synchronous copy on `stream` into *status_out (host).  Clears it when
 * `clear` is non-zero. */
int dg_read_device_status(const void *workspace, int *status_out, int clear, void *stream);

/* ------------------------------------------------------------------------ */
/* Canvas attention.                                                         */
/* "DiffusionGemma Lab" section 2 item 6 and "Parallel Denoising ..." section */
/* "Finding": the decoder attends bidirectionally across the canvas (no mask) */
/* and to the causal encoder's KV cache.  For batch b, canvas position i and  */
/* query head h, with kv head g = h / (Hq / Hkv):                             */
/*   out[b,i,h,:] = softmax_j(scale * q[b,i,h,:] . K_j) V_j,                  */
/* keys j running over the P cached rows k_prefix[b,:,g,:] followed by the L  */
/* canvas rows k_canvas[b,:,g,:] (same for V).                                 */
/* Layouts: q, out [B, L, Hq, D]; k_prefix, v_prefix [B, P, Hkv, D];          */
/*          k_canvas, v_canvas [B, L, Hkv, D]; all bf16.                       */
/* bf16 inputs, fp32 accumulation and softmax, bf16 output.                   */
/* Supported: D in {128, 256}; Hq % Hkv == 0 and Hq/Hkv a power of two <= 16; */
/* 1 <= L; 0 <= P; B >= 1.  P == 0 is allowed (k_prefix/v_prefix may be NULL).*/
/* ------------------------------------------------------------------------ */
size_t dg_canvas_attn_workspace(int B, int L, int P, int Hq, int Hkv, int D);
int dg_canvas_attn(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                   const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *out,
                   int B, int L, int P, int Hq, int Hkv, int D, float scale,
                   void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* Encoder cache append.                                                     */
/* "Parallel Denoising From an Autoregressive Checkpoint", section           */
/* "Finding": after a block is committed, the causal encoder runs once more  */
/* over it and extends its append-only KV cache, which the next block's      */
/* canvas then attends to.  This call (1) copies the block's keys / values   */
/* k_new, v_new [B, L, Hkv, D] into rows P .. P+L-1 of the caches k_cache,   */
/* v_cache [B, P_max, Hkv, D] (rows 0 .. P-1 hold the earlier tokens) and    */
/* (2) computes the block's causal attention: for canvas position i,         */
/*   out[b,i,h,:] = softmax_j(scale * q[b,i,h,:] . K_j) V_j over the P cached */
/* rows and the block's rows 0 .. i.  q, out [B, L, Hq, D]; all bf16;         */
/* P_max >= P + L.  After the call the caches hold P + L tokens.  Same        */
/* kernels, supported shapes and workspace rules as dg_canvas_attn; the       */
/* caches are written in stream order before the attention reads them.       */
/* ------------------------------------------------------------------------ */
size_t dg_encoder_append_workspace(int B, int L, int P, int Hq, int Hkv, int D);
int dg_encoder_append(const uint16_t *q, uint16_t *k_cache, uint16_t *v_cache, int P, int P_max,
                      const uint16_t *k_new, const uint16_t *v_new, uint16_t *out, int B, int L,
                      int Hq, int Hkv, int D, float scale, void *workspace,
                      size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------ */
/* One denoising step after the decoder body: LM head -> per-position        */
/* entropy, Gumbel-max sample and argmax -> entropy-bounded acceptance and    */
/* uniform renoise -> adaptive stop test.                                     */
/*                                                                            */
/* "DiffusionGemma Lab" section 2 items 2, 3 and 5; "Parallel Denoising ..."  */
/* section "Finding", bullets "Entropy-bounded acceptance" and "Adaptive      */
/* stopping".  Per canvas position (row r = b*L + i):                         */
/*   logits = hidden[r,:] . w          (bf16 in, fp32 accumulate; never       */
/*                                      written to memory)                    */
/*   entropy[r] = H(softmax(logits / T)) in nats                              */
/*   argmax[r]  = argmax logits (ties -> lowest vocabulary index)             */
/*   sample[r]  = argmax_v fp32(fmaf(logit_v, fp32(1/T), G_v)), G_v the       */
/*                standard Gumbel variate -ln(-ln u) of Philox4x32-10 word    */
/*                (v & 3) of counter (v >> 2, r, step, 0), key = seed         */
/*   per canvas: sort positions by (entropy, position) ascending; commit the  */
/*   largest prefix whose entropies, minus its largest one, sum (fp64) to     */
/*   <= entropy_bound (always >= 1): canvas[r] = sample[r], accepted[r] = 1;  */
/*   every other position is redrawn: canvas[r] = (x * V) >> 32 with x word 0 */
/*   of counter (0, r, step, 1).                                              */
/*   stop[b] = step >= 1 && argmax == prev_argmax over the canvas &&          */
/*             mean entropy < stop_threshold; then prev_argmax <- argmax.     */
/* Layouts: hidden [B*L, d] bf16; w [d, V] bf16 (vocabulary contiguous), or */
/* with w_layout = DG_W_PACKED the same weight as dg_pack_lm_weight writes   */
/* it (then only the 2-SM LM-head kernels run: w is read as one 16 KB        */
/* stretch per 128 columns and 64 hidden dimensions).                        */
/* Supported: d % 64 == 0, 64 <= d <= 16384; V % 8 == 0, 64 <= V < 2^31;      */
/* 1 <= L <= 1024; B >= 1.                                                    */
/* ------------------------------------------------------------------------ */
#define DG_W_ROWMAJOR 0     /* w [d, V]                                        */
#define DG_W_PACKED 1       /* w as dg_pack_lm_weight writes it                */
typedef struct dg_step_params {
    int B;                  /* canvases in the batch                          */
    int L;                  /* canvas length (256)                            */
    int d;                  /* hidden size                                    */
    int V;                  /* vocabulary size                                */
    double temperature;     /* T of this step, > 0 (1/T is rounded to fp32)   */
    float entropy_bound;    /* b (0.1)                                        */
    float stop_threshold;   /* mean-entropy stop threshold (0.005)            */
    int step;               /* step index k (Philox counter; k >= 1 arms stop)*/
    uint64_t seed;          /* Philox key                                     */
    int w_layout;           /* DG_W_ROWMAJOR (0) or DG_W_PACKED               */
} dg_step_params;

/* The LM-head weight in the layout the 2-SM kernels stream fastest: the      */
/* columns in tiles of 128, each tile's d rows of 128 values contiguous:      */
/*   w_packed[t][k][c] = w[k][128 t + c]   (c < 128, t < ceil(V / 128)),      */
/* zero where 128 t + c >= V.  A tile of 128 columns by 64 hidden dimensions  */
/* is then one contiguous 16 KB stretch of memory instead of 64 rows of 256   */
/* bytes a row of w apart.  w [d, V] bf16 (device), w_packed of               */
/* dg_lm_weight_packed_bytes(d, V) bytes (device, caller-owned, not          */
/* overlapping w); one kernel launch on `stream`.  Returns DG_ERR_INVALID_ARG */
/* for null pointers or d, V outside the step's supported range, else        */
/* DG_ERR_CUDA on a launch failure.  A layout choice only: the step's         */
/* results are the same bit for bit with either layout.                       */
size_t dg_lm_weight_packed_bytes(int d, int V);
int dg_pack_lm_weight(const uint16_t *w, int d, int V, uint16_t *w_packed, void *stream);

typedef struct dg_step_io {
    int32_t *canvas;        /* [B*L] in/out: current canvas tokens            */
    int32_t *prev_argmax;   /* [B*L] in/out: argmax of the previous step      */
    int32_t *argmax;        /* [B*L] out                                      */
    int32_t *sample;        /* [B*L] out                                      */
    float *entropy;         /* [B*L] out, nats                                */
    uint8_t *accepted;      /* [B*L] out, 1 = committed this step             */
    int32_t *n_accepted;    /* [B]   out                                      */
    float *mean_entropy;    /* [B]   out                                      */
    int32_t *stop;          /* [B]   out, 1 = stop                            */
} dg_step_io;

size_t dg_denoise_step_workspace(const dg_step_params *p);
int dg_denoise_step(const uint16_t *hidden, const uint16_t *w, const dg_step_params *p,
                    const dg_step_io *io, void *workspace, size_t workspace_bytes,
                    void *stream);

/* The whole step in one call: dg_canvas_attn (the canvas's attention over   */
/* [cache ; canvas], into attn_out) and dg_denoise_step (the LM head, sampler, */
/* acceptance and stop test on the given hidden states).  In this step the    */
/* two read different inputs, so the attention runs on a second stream the     */
/* library forks from `stream` and joins back into it (the call's work on      */
/* `stream` ends when both have); when the attention is short on few CTAs    */
/* (its key splits capped at an eighth of the SMs, else a sixth, leave at     */
/* most 6 key tiles per CTA) the LM head is planned on the SMs it leaves --   */
/* on fewer of them set aside when that gives the LM head more CTAs and the   */
/* attention still at most 12 key tiles per reserved SM.                      */
/* The second stream is one per device, shared by all calls: calls on         */
/* different streams, or from several host threads (the library enqueues a    */
/* call's fork, launches and join under a lock), are correct but their        */
/* attentions run one after another.                                          */
/* Arguments as the two calls (B, L of p; q / out [B, L, Hq, D]; caches       */
/* [B, P, Hkv, D]); one workspace of dg_canvas_step_workspace bytes: the     */
/* step's first (its status word at the start), then the attention's from    */
/* offset round_up(dg_denoise_step_workspace(p), 256) (its own status word). */
/* Errors as the two calls.  Capturable (the fork and join become graph       */
/* edges).                                                                    */
size_t dg_canvas_step_workspace(const dg_step_params *p, int P, int Hq, int Hkv, int D);
int dg_canvas_step(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                   const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *attn_out, int P,
                   int Hq, int Hkv, int D, float scale, const uint16_t *hidden, const uint16_t *w,
                   const dg_step_params *p, const dg_step_io *io, void *workspace,
                   size_t workspace_bytes, void *stream);

/* The whole step with the E4M3 LM head (dg_denoise_step_fp8) or with the     */
/* self-conditioning read-out (dg_denoise_step_sc) in place of               */
/* dg_denoise_step: the canvas attention on the library's second stream,     */
/* forked from `stream` and joined back into it, beside that step on         */
/* `stream`; no SMs are set aside for the attention.  Arguments and errors   */
/* as dg_canvas_attn and the step they pair with; one workspace of the       */
/* matching *_workspace bytes: the step's first (its status word at the      */
/* start), the attention's from offset round_up(step workspace, 256).        */
/* Same results as the two calls, bit for bit.                               */
size_t dg_canvas_step_fp8_workspace(const dg_step_params *p, int P, int Hq, int Hkv, int D);
int dg_canvas_step_fp8(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                       const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *attn_out,
                       int P, int Hq, int Hkv, int D, float scale, const uint16_t *hidden,
                       const uint8_t *w8t, const float *w_scale, const dg_step_params *p,
                       const dg_step_io *io, void *workspace, size_t workspace_bytes,
                       void *stream);
size_t dg_canvas_step_sc_workspace(const dg_step_params *p, int P, int Hq, int Hkv, int D);
int dg_canvas_step_sc(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                      const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *attn_out,
                      int P, int Hq, int Hkv, int D, float scale, const uint16_t *hidden,
                      const uint16_t *w, const uint16_t *sc_table, const dg_step_params *p,
                      const dg_step_io *io, float *sc_out, void *workspace,
                      size_t workspace_bytes, void *stream);

/* dg_denoise_step for callers that cannot allocate device memory (an engine  */
/* that owns every byte through its own pool, code that runs where allocation */
/* is not allowed): no workspace argument.  The pages have no counterpart;    */
/* this is a deployment convenience.  Same kernels, same results (w in either */
/* layout of p->w_layout); their                                              */
/* scratch lives in one 8 MiB array inside the library's device memory,      */
/* held by every GPU that loads the library until the process exits.         */
/* Limit: steps needing more than 8 MiB of scratch (256 B + 7 x 4 B x units  */
/* x B*L + 4 B x B + 4 B x B*L, each term but the first rounded up to 256 B; */
/* units = the LM-head plan's CTAs, or clusters for kinds 2/3; every step    */
/* with B*L <= 1968 fits on a 152-SM GB300) return DG_ERR_UNSUPPORTED.  The first call on a device */
/* sets up the array's address (cudaGetSymbolAddress) and clears its status  */
/* header: make it before any stream capture.  All calls share the array;    */
/* calls that overlap on the GPU race -- order them on one stream.  Calls no */
/* cudaMalloc/cudaFree.  Device-side errors of this path are read with       */
/* dg_noalloc_read_device_status, not dg_read_device_status.                 */
int dg_denoise_step_noalloc(const uint16_t *hidden, const uint16_t *w, const dg_step_params *p,
                            const dg_step_io *io, void *stream);

/* The device status word of dg_denoise_step_noalloc's scratch array (0 or a  */
/* DG_ERR_* code recorded by its kernels), read with a synchronous copy on    */
/* `stream` into *status_out (host); clear != 0 resets it.  Allocates        */
/* nothing.  Errors: DG_ERR_INVALID_ARG (null status_out), DG_ERR_CUDA.      */
int dg_noalloc_read_device_status(int *status_out, int clear, void *stream);

/* ------------------------------------------------------------------------ */
/* dg_denoise_step with the self-conditioning read-out folded into the LM    */
/* head.  "Parallel Denoising From an Autoregressive Checkpoint", section    */
/* "Finding": a 7.8M-parameter self-conditioning block feeds the previous    */
/* step's prediction back into the model, and its matmul runs in the         */
/* sampling stage next to the full-vocabulary softmax.  The pages give no   */
/* formula; this library reads the fed-back prediction as the expected       */
/* embedding under the step's sampling distribution:                         */
/*   sc_out[r, j] = sum_v softmax(logits[r] / T)_v sc_table[v, j],  j < 32   */
/* (V x 30 = 7.86M parameters at V = 262144; pad the table's rows with zero  */
/* columns to 32).  The weights 2^(t - m) of each 16-column chunk are rounded */
/* to bf16 and multiplied with the table on the tensor cores (fp32           */
/* accumulation); softmax statistics and the read-out sums are fp32; the      */
/* logits are never stored.  Turning sc_out into the next step's hidden      */
/* states is the decoder body's work.  Layouts: sc_table [V, 32] bf16         */
/* (device, 16-byte aligned), sc_out [B*L, 32] fp32 (device, 16-byte          */
/* aligned); the rest as dg_denoise_step.  Always runs the 2-SM LM-head       */
/* kernel.  Every other output as dg_denoise_step.  Errors as                 */
/* dg_denoise_step.                                                           */
/* ------------------------------------------------------------------------ */
size_t dg_denoise_step_sc_workspace(const dg_step_params *p);
int dg_denoise_step_sc(const uint16_t *hidden, const uint16_t *w, const uint16_t *sc_table,
                       const dg_step_params *p, const dg_step_io *io, float *sc_out,
                       void *workspace, size_t workspace_bytes, void *stream);
/* Its LM-head kernel alone (partial states and read-out parts left in the   */
/* workspace; for timing).                                                    */
int dg_lm_head_fold_sc(const uint16_t *hidden, const uint16_t *w, const uint16_t *sc_table,
                       const dg_step_params *p, void *workspace, size_t workspace_bytes,
                       void *stream);

/* ------------------------------------------------------------------------ */
/* Mixture-of-experts FFN over the canvas hidden states (the decoder body's  */
/* largest per-step cost).  "DiffusionGemma: When the LLM Stops Writing Left  */
/* to Right", section "What DiffusionGemma Actually Is": 128 experts, top-8  */
/* routing and one shared expert; "Parallel Denoising From an Autoregressive */
/* Checkpoint", section "Finding": a canvas forward touches about 84 distinct */
/* experts per layer.  The pages give no formulas; this library computes,    */
/* per row t of x:                                                           */
/*   l = x_t . w_router^T (fp32);  S_t = the top_k experts by l (ties to the */
/*   lower index), gates g = softmax(l[S_t]);                                */
/*   FFN_e(x) = (gelu_tanh(x . w_gate[e]^T) * (x . w_up[e]^T)) . w_down[e]^T,  */
/*   the product of the first two rounded to bf16 before the last matmul;    */
/*   out_t = FFN_E(x_t) + sum_j g_j FFN_{S_t[j]}(x_t)  (expert E = shared).   */
/* bf16 operands, fp32 accumulation (tensor cores), fp32 output.  Layouts    */
/* (bf16, K-major "weights as rows"): x [M, d]; w_router [E, d]; w_gate,      */
/* w_up [E + 1, f, d]; w_down [E + 1, d, f] (index E = the shared expert);   */
/* out [M, d] fp32.  experts_out [M, top_k] int32 and gates_out [M, top_k]   */
/* fp32 receive the routing when not NULL.  Only the experts some row picks */
/* are read.  Supported: 1 <= M <= 2048; d, f multiples of 128, <= 16384;     */
/* 1 <= top_k <= min(8, E), E <= 128.  16-byte aligned pointers.  Errors as  */
/* dg_denoise_step; device-side waits report through the workspace status.  */
/* ------------------------------------------------------------------------ */
typedef struct dg_moe_params {
    int M;          /* canvas rows (B * L)                                    */
    int d;          /* hidden size                                            */
    int f;          /* FFN width of every expert                              */
    int n_experts;  /* routed experts E (the shared one is extra)             */
    int top_k;      /* experts per row                                        */
} dg_moe_params;

size_t dg_moe_ffn_workspace(const dg_moe_params *p);
int dg_moe_ffn(const uint16_t *x, const uint16_t *w_router, const uint16_t *w_gate,
               const uint16_t *w_up, const uint16_t *w_down, float *out, int32_t *experts_out,
               float *gates_out, const dg_moe_params *p, void *workspace, size_t workspace_bytes,
               void *stream);

/* ------------------------------------------------------------------------ */
/* The denoising loop of one block (batch of B independent canvases).        */
/* "DiffusionGemma Lab" section 2 items 1-5; "Parallel Denoising ..."         */
/* section "Finding" (temperature annealing, adaptive stopping, N = 48).      */
/* Initialises canvas[r] = (x * V) >> 32, x word 0 of Philox counter          */
/* (0, r, 0, 2); then for k = 0 .. max_steps-1 runs dg_denoise_step with      */
/* T_k = t_start + (t_end - t_start) * k / (max_steps - 1) (computed in fp64) */
/* on hidden_steps + k * hidden_step_stride, until every canvas has stopped.  */
/* A canvas that stops keeps its canvas and argmax from that step.  The loop  */
/* runs on the device as one CUDA graph with a conditional while node; the    */
/* host waits only at the end.  The library keeps the instantiated graph of   */
/* each distinct (pointers, shapes, params incl. the seed, block params, W    */
/* layout, LM-head plan, producer) and replays it on a repeated call; it      */
/* keeps at most 64, dropping the least recently used (the call that drops   */
/* one waits on the host for that graph's last launch to complete before it  */
/* frees it).  A call with a new key captures and instantiates a graph on     */
/* the host before it launches.                                               */
/* hidden_steps: device bf16, hidden_step_stride elements apart per step (0 = */
/* the same hidden states every step); the decoder body that would produce    */
/* them is outside this library.                                              */
/* ------------------------------------------------------------------------ */
typedef struct dg_block_params {
    int max_steps;              /* N (48)                                     */
    double t_start;             /* 0.8                                        */
    double t_end;               /* 0.4                                        */
    int64_t hidden_step_stride; /* elements between consecutive steps         */
} dg_block_params;

typedef struct dg_block_io {
    int32_t *canvas;            /* [B*L] out: final canvas tokens             */
    int32_t *argmax;            /* [B*L] out: the block output                */
    int32_t *steps_taken;       /* [B]   out                                  */
    float *mean_entropy;        /* [B]   out: at the last step taken          */
    int32_t *n_accepted_hist;   /* [max_steps*B] out, may be NULL             */
} dg_block_io;

size_t dg_generate_block_workspace(const dg_step_params *p, const dg_block_params *bp);
int dg_generate_block(const uint16_t *hidden_steps, const uint16_t *w,
                      const dg_step_params *p, const dg_block_params *bp,
                      const dg_block_io *io, void *workspace, size_t workspace_bytes,
                      void *stream);

/* The block loop with the decoder body inside it.  "DiffusionGemma Lab",     */
/* section 2 items 1-5: every step re-runs the decoder on the current canvas  */
/* and samples from its logits.  produce_hidden enqueues, on `stream`, the    */
/* work that writes the hidden states [B*L, d] (bf16) of the step into        */
/* hidden_buf; the loop then runs dg_denoise_step on them.  The loop is one   */
/* CUDA graph whose body is captured once per (shapes, pointers, callback,    */
/* user) and replayed for every step on the device, so the callback is        */
/* invoked while `stream` is being captured (once per distinct key, not once  */
/* per step): it must enqueue only capturable work (kernel launches, async    */
/* copies; no allocation, no synchronisation) and read the step index k from */
/* *step (device int32, valid when its work runs) and the current canvas      */
/* from canvas (device [B*L] int32, the tokens the step starts from).  It     */
/* returns DG_OK or an error, which the call returns.  Everything else as     */
/* dg_generate_block (hidden_step_stride is ignored).                        */
typedef int (*dg_hidden_fn)(const int32_t *step, const int32_t *canvas, uint16_t *hidden_out,
                            void *stream, void *user);
int dg_generate_block_fn(dg_hidden_fn produce_hidden, void *user, uint16_t *hidden_buf,
                         const uint16_t *w, const dg_step_params *p, const dg_block_params *bp,
                         const dg_block_io *io, void *workspace, size_t workspace_bytes,
                         void *stream);

/* Producers for dg_generate_block_fn (user points to the struct named).     */
/* dg_hidden_from_steps: hidden_out = hidden_steps + k * step_stride, n       */
/* elements (the hidden states of every step computed ahead, the same loop as */
/* dg_generate_block).                                                        */
typedef struct dg_hidden_steps {
    const uint16_t *hidden_steps;   /* device bf16                            */
    int64_t step_stride;            /* elements between steps                 */
    int64_t n;                      /* elements per step (B * L * d)          */
} dg_hidden_steps;
int dg_hidden_from_steps(const int32_t *step, const int32_t *canvas, uint16_t *hidden_out,
                         void *stream, void *user);
/* dg_hidden_embed_add: hidden_out[r, j] = bf16(base_k[r, j] + table[canvas[r], */
/* j]) with base_k = base + k * base_step_stride (fp32 sum, nearest even): a  */
/* stand-in decoder whose output depends on the canvas being denoised (token  */
/* ids are clamped to [0, V)).                                                */
typedef struct dg_hidden_embed {
    const uint16_t *base;           /* device bf16 [rows, d] per step         */
    int64_t base_step_stride;       /* elements between steps (0: one base)   */
    const uint16_t *table;          /* device bf16 [V, d]                     */
    int rows, d, V;
} dg_hidden_embed;
int dg_hidden_embed_add(const int32_t *step, const int32_t *canvas, uint16_t *hidden_out,
                        void *stream, void *user);

/* ------------------------------------------------------------------------ */
/* Entry points that run one stage of the step on given inputs, through the  */
/* same device code as dg_denoise_step (for checking each stage alone).      */
/* ------------------------------------------------------------------------ */

/* The step of dg_denoise_step with fp32 logits [B*L, V] read from memory in  */
/* place of hidden . w.  Same params/io; p->d is ignored. */
size_t dg_sampler_workspace(const dg_step_params *p);
int dg_sampler_from_logits(const float *logits, const dg_step_params *p, const dg_step_io *io,
                           void *workspace, size_t workspace_bytes, void *stream);

/* The first kernel of dg_denoise_step alone: the LM-head GEMM with its      */
/* fused entropy / Gumbel-max / argmax epilogue, leaving the per-position     */
/* partial states in the workspace (no combine, acceptance or stop).  Same    */
/* arguments and workspace size as dg_denoise_step; io is not needed.         */
int dg_lm_head_fold(const uint16_t *hidden, const uint16_t *w, const dg_step_params *p,
                    void *workspace, size_t workspace_bytes, void *stream);

/* Number of kernels this library has launched (or enqueued into a stream    */
/* capture) in this process so far.                                           */
uint64_t dg_kernel_launches(void);

/* The LM-head launch dg_denoise_step would make on the current device for    */
/* rows = B*L canvas positions, hidden size d and vocabulary V (no launch),  */
/* with W [d, V] in its row-major layout (a packed W keeps the step on the   */
/* kinds 2 and 3; the FP8 step runs kind 2/3 with 12 epilogue warps).       */
/* *kind: 0 = single-CTA kernel, 2 = 2-CTA cluster issuing 2-SM UMMAs,      */
/* 3 = the kind-2 kernel on a schedule of bn-column tiles whose adjacent     */
/* pairs run as one tile of 2 bn columns (kind 1 is not used); *bn:          */
/* vocabulary columns per (schedule) tile; *ctas: CTAs launched;             */
/* *epilogue_warps: the kind-2/3 kernel's epilogue warps (8 for a single     */
/* 256-row block, else 16; 0 for kind 0).  Any output pointer                */
/* may be NULL.                                                               */
/* Returns DG_ERR_INVALID_ARG / DG_ERR_UNSUPPORTED for shapes the step        */
/* rejects, DG_ERR_CUDA without a device. */
int dg_lm_head_plan(int rows, int d, int V, int *kind, int *bn, int *ctas, int *epilogue_warps);

/* The launches dg_canvas_step would make for these arguments (same meaning  */
/* as there) on a GPU with `sms` SMs, without launching anything.  sms > 0   */
/* (at most 256) plans for that SM count and touches no device, so it runs   */
/* on a host without a GPU; sms <= 0 takes the current device's count        */
/* (DG_ERR_CUDA without a device).  The planner's environment overrides      */
/* (DG_ATTN_*, DG_LM_*) apply as in the step.                                 */
typedef struct dg_canvas_step_plan_info {
    int attn_reserved_sms;  /* SMs set aside for the attention; 0: it shares */
                            /* the GPU with the LM head                        */
    int attn_pair;          /* 1: 2-CTA clusters issuing 2-SM UMMAs (adjacent */
                            /* 128-row query tiles), 0: one CTA per tile      */
    int attn_ctas;          /* CTAs of the attention kernel                    */
    int attn_splits;        /* key splits per query tile (> 1: a merge kernel  */
                            /* follows)                                         */
    int attn_key_tiles;     /* key tiles per split, at most                    */
    int attn_key_tile;      /* keys per key tile                               */
    int lm_kind;            /* as *kind of dg_lm_head_plan                     */
    int lm_bn;              /* vocabulary columns per (schedule) tile          */
    int lm_ctas;            /* CTAs of the LM-head kernel                      */
    int lm_tiles;           /* tiles of its schedule                           */
    int lm_epilogue_warps;  /* as *epilogue_warps of dg_lm_head_plan           */
    int lm_sms;             /* SMs the LM head was planned on                  */
} dg_canvas_step_plan_info;
/* Errors: DG_ERR_INVALID_ARG for a NULL p or out, invalid params or sms     */
/* above 256; DG_ERR_UNSUPPORTED for shapes dg_canvas_step rejects.  *out is */
/* written only on DG_OK. */
int dg_canvas_step_plan(const dg_step_params *p, int P, int Hq, int Hkv, int D, int sms,
                        dg_canvas_step_plan_info *out);

/* ------------------------------------------------------------------------ */
/* FP8 (E4M3) LM head.  The pages quote their throughput for an FP8 model     */
/* ("DiffusionGemma Lab" section 1; "Parallel Denoising From an              */
/* Autoregressive Checkpoint", section "Finding"); E4M3 is the OCP FP8       */
/* format (bias 7, no infinities, largest finite 448).  The pages do not fix */
/* the scaling granularity; this library takes one fp32 scale per canvas row  */
/* of the hidden states and one per vocabulary column of W.                   */
/* Quantising a row x[0..n): amax = max |x_j|; amax == 0: codes 0, scale 1;   */
/* else inv = fp32(448 / amax), scale = fp32(amax / 448) and code_j = the    */
/* E4M3 value nearest fp32(x_j * inv) (ties to even, saturated at +-448).    */
/* The row stands for decode(code_j) * scale.                                 */
/* ------------------------------------------------------------------------ */

/* x [rows, cols] bf16 (device) -> codes [rows, cols] u8 and scale [rows] f32 */
/* (device, caller-owned).  Any alignment.  Errors: DG_ERR_INVALID_ARG for    */
/* null pointers or sizes < 1; DG_ERR_CUDA if the launch fails.               */
int dg_quantize_rows_e4m3(const uint16_t *x, int64_t rows, int cols, uint8_t *codes,
                          float *scale, void *stream);

/* W [d, V] bf16 (vocabulary contiguous, device) -> w8t [V, d] u8 (the       */
/* transposed codes, each vocabulary column quantised as one row) and        */
/* scale [V] f32 (device, caller-owned).  A load-time conversion of the      */
/* model's weight (3 launches).  Errors as dg_quantize_rows_e4m3.            */
int dg_quantize_weight_e4m3(const uint16_t *w, int d, int V, uint8_t *w8t, float *scale,
                            void *stream);

/* dg_denoise_step with the LM head on E4M3 operands: the hidden states are  */
/* quantised per row inside the step (into the workspace), the weight comes  */
/* quantised by dg_quantize_weight_e4m3, and                                  */
/*   logit[r, v] = (sum_k dec(x8[r,k]) dec(w8t[v,k])) * sx[r] * w_scale[v]   */
/* (fp32 accumulation on the tensor cores, then two fp32 products); the      */
/* sampler, acceptance and stop test are dg_denoise_step's.  Layouts: hidden */
/* [B*L, d] bf16; w8t [V, d] u8; w_scale [V] f32; all 16-byte aligned.        */
/* Supported: d % 128 == 0, 128 <= d <= 16384; V, L, B as dg_denoise_step.   */
/* Errors as dg_denoise_step.                                                 */
size_t dg_denoise_step_fp8_workspace(const dg_step_params *p);
int dg_denoise_step_fp8(const uint16_t *hidden, const uint8_t *w8t, const float *w_scale,
                        const dg_step_params *p, const dg_step_io *io, void *workspace,
                        size_t workspace_bytes, void *stream);

/* The quantisation of the hidden states and the FP8 LM-head kernel of       */
/* dg_denoise_step_fp8 alone (partial states left in the workspace).         */
int dg_lm_head_fold_fp8(const uint16_t *hidden, const uint8_t *w8t, const float *w_scale,
                        const dg_step_params *p, void *workspace, size_t workspace_bytes,
                        void *stream);

/* Acceptance, renoise and stop test alone on given entropy/sample/argmax     */
/* [B*L] (device).  Writes canvas, accepted, n_accepted, stop, mean_entropy   */
/* and prev_argmax of io; io->entropy/sample/argmax are not used. */
int dg_accept_renoise(const float *entropy, const int32_t *sample, const int32_t *argmax,
                      const dg_step_params *p, const dg_step_io *io, void *workspace,
                      size_t workspace_bytes, void *stream);

/* Standard Gumbel variates of vocabulary entries v0 .. v0+n-1 for (row, step) */
/* as the sampler draws them (device float[n]). */
int dg_gumbel_fill(uint64_t seed, uint32_t row, uint32_t step, uint32_t v0, int n,
                   float *out, void *stream);

/* The sampler's fp32 natural logarithm applied to x[0..n) (device arrays).   */
int dg_logf_eval(const float *x, float *y, int n, void *stream);

/* The failure path of the library's bounded device waits, on its own (the   */
/* pages describe no failure handling; this is a check of the library).  One */
/* warp allocates 32 TMEM columns, waits on an mbarrier that nothing ever     */
/* arrives on, gives up after limit_ns nanoseconds of global time, records  */
/* DG_ERR_TIMEOUT in the workspace's status word, frees its TMEM and         */
/* returns -- the way every kernel of the library winds down when a wait     */
/* runs out.  The context stays usable.  limit_ns in [1000, 1e9].  Errors:   */
/* DG_ERR_WORKSPACE (workspace missing or < 256 B), DG_ERR_INVALID_ARG,      */
/* DG_ERR_ALIGNMENT, DG_ERR_CUDA.                                            */
int dg_wait_timeout_probe(void *workspace, size_t workspace_bytes, uint64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
