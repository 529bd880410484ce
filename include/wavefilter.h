/*
 * wavefilter.h — C ABI of the GB300 (sm_103a) WaveFilter KV-filtering path.
 *
 * Method: "WaveFilter: Enhancing the Long-Context Capability of Diffusion
 * LLMs via Wavelet-Guided KV Cache Filtering" (arXiv 2606.00724).  One call
 * chain filters the cached prompt keys of one layer at one denoising step
 * t > 1 and attends over the resulting sparse cache:
 *
 *   wf_dwt_lowpass        §2.2 eq. (5) pyramid, §3.1: Haar DWT of K~[I_p]
 *   wf_score_topk         Fig. 2(c): query/low-frequency scoring + Top-K
 *   wf_recursive_filter   Fig. 2(d), §3 overview: coarse-to-fine refinement
 *   wf_sparse_gather_attn §2.1 eq. (3) over the sparse cache S ∪ I_g
 *   wf_step               all four, in order, on one stream
 *
 * and the cache writes around it:
 *
 *   wf_cache_init         §2.1 eq. (2) at t = 1, plus A_L of the prompt keys
 *   wf_cache_update       §2.1 eq. (4) at t > 1 (generation rows)
 *   wf_cache_scatter      §2.1 eq. (4) over any position set, with A_L repair
 *
 * and, for wavelet bases longer than the Haar pair (§3.1 leaves psi open):
 *
 *   wf_daubechies_lowpass  the extremal-phase Daubechies low-pass filters
 *   wf_dwt_lowpass_basis   the pyramid A_1..A_L of such a basis
 *   wf_step_basis          the whole step with such a basis
 *
 * Readings fixed where the pages are silent: orthonormal Haar filters
 * g = [1/√2, 1/√2] on 0-based pairs (2n, 2n+1), so coarse position p at
 * level j covers tokens [p·2^j, (p+1)·2^j); the score of a candidate is its
 * attention mass (per-query softmax of Q·A_j/√d over the current candidate
 * set, summed over the queries); candidates at level j < L are the children
 * {2p, 2p+1} of the level-(j+1) survivors; Top-K prefers the larger score
 * and, on equal scores, the lower position; no attention mask.
 *
 * Shapes (row-major, contiguous; U = batch·heads independent units):
 *   Kp, Vp : [batch, heads, n_prompt, head_dim]   prompt keys/values  (I_p)
 *   Kg, Vg : [batch, heads, n_gen,    head_dim]   generation keys/values (I_g)
 *   Q      : [batch, heads, n_gen,    head_dim]   generation-block queries
 * Element type of Q/K/V: dims.dtype (WF_BF16 or WF_F32).  All arithmetic
 * accumulates in fp32; every float output is fp32.
 *
 * Ownership and execution: the caller owns every buffer.  All pointers are
 * DEVICE pointers except those documented as host (k_per_level, dims).
 * Every device pointer must be 16-byte aligned.  The library never allocates
 * device memory and never synchronises: each entry point validates its
 * arguments on the host, then enqueues kernels on `stream` (a cudaStream_t;
 * NULL = legacy default stream) and returns.  On any validation error
 * nothing is enqueued.  Launch failures are reported as WF_ERR_CUDA.
 * Data-dependent faults found on the device (an index outside [0, n_prompt)
 * or a duplicate survivor) never cause an out-of-bounds access: the offending
 * entry is skipped and a code is recorded in the workspace status word,
 * readable with wf_read_device_status().
 *
 * Determinism: identical inputs give bit-identical outputs (fixed reduction
 * orders, no floating-point atomics).
 */
#ifndef WAVEFILTER_H_
#define WAVEFILTER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum {
  WF_OK = 0,
  WF_ERR_NULL = 1,          /* a required pointer is NULL                        */
  WF_ERR_SHAPE = 2,         /* inconsistent sizes / per-level k (see wf_step)    */
  WF_ERR_UNSUPPORTED = 3,   /* head_dim not 64/128, unknown dtype, n_gen > 64    */
  WF_ERR_WORKSPACE = 4,     /* workspace smaller than wf_workspace_bytes()       */
  WF_ERR_CUDA = 5,          /* a CUDA launch or query failed                     */
  WF_ERR_DEVICE_CHECK = 6,  /* a device-side check failed (device status word)   */
  WF_ERR_ALIGNMENT = 7      /* a device pointer is not 16-byte aligned           */
};

/* Element types of Q, K, V. */
enum { WF_BF16 = 0, WF_F32 = 1 };

/* Device status word codes (bit flags, OR-ed by the kernels). */
enum {
  WF_DEV_OK = 0,
  WF_DEV_BAD_INDEX = 1,      /* an index outside [0, n_prompt) (or its level range) */
  WF_DEV_DUP_INDEX = 2,      /* a duplicate coarse survivor                         */
  WF_DEV_WAIT_TIMEOUT = 4    /* a bounded wait on an asynchronous copy gave up      */
};

/* Limits of this build. */
#define WF_MAX_LEVELS 12
#define WF_MAX_GEN 64

/* Problem dimensions (host struct, read during the call only).
 *   batch, heads       : U = batch·heads independent (sequence, head) units
 *   n_prompt           : N_p = |I_p|, must be a multiple of 2^levels
 *   n_gen              : G = |I_g| = number of generation-block queries, 1..64
 *   head_dim           : d ∈ {64, 128}
 *   levels             : L, 1..12 (Haar levels; A_L has N_p/2^L positions)
 *   dtype              : WF_BF16 or WF_F32 (element type of Q/K/V) */
typedef struct {
  int32_t batch, heads, n_prompt, n_gen, head_dim, levels, dtype;
} wf_dims;

/* Human-readable name of a status code (static string, never NULL). */
const char* wf_status_string(int status);

/* Name and description of the last CUDA error that made an entry point of
 * this thread return WF_ERR_CUDA (thread-local; "no error" initially). */
const char* wf_last_error_string(void);

/* Default per-level survivor counts (host helper; not on the device path).
 * k_out[j], j = 0..levels: k_L = ceil(2·budget / 2^L) capped at N_p/2^L,
 * k_j = min(2^(L-j)·k_L, N_p/2^j) for 0 < j < L, k_0 = budget.
 * Returns WF_ERR_SHAPE if budget < 1 or n_prompt is not a multiple of 2^L. */
int wf_default_k_per_level(int32_t n_prompt, int32_t levels, int32_t budget,
                           int32_t* k_out);

/* Bytes of device workspace wf_step (and each stage) needs for these sizes.
 * k_per_level: host array of levels+1 entries (see wf_recursive_filter).
 * Stores the byte count in *bytes.  Errors: WF_ERR_NULL/SHAPE/UNSUPPORTED. */
int wf_workspace_bytes(const wf_dims* dims, const int32_t* k_per_level,
                       size_t* bytes);

/* Number of kernel launches one wf_step call makes for these sizes on the
 * current device: 1 where the level-L approximation is computed inside the
 * path kernel (per-CTA slice of at most 64 coarse positions whose spans fit
 * the streaming ring), else 2 (a separate streaming DWT launch first).
 * Stores it in *launches.  Host only; launches nothing.
 * Errors: WF_ERR_NULL/SHAPE/UNSUPPORTED, as wf_workspace_bytes. */
int wf_step_launch_count(const wf_dims* dims, const int32_t* k_per_level,
                         int32_t* launches);

/* Where the token-level logits of the recursive filter are kept (wf_plan). */
enum {
  WF_LOGITS_SHARED = 0,          /* in shared memory                              */
  WF_LOGITS_WORKSPACE = 1,       /* written to the workspace and read back        */
  WF_LOGITS_TENSOR_MEMORY = 2,   /* in the accumulators' tensor memory            */
  WF_LOGITS_RECOMPUTED = 3       /* recomputed from the key rows for each pass    */
};

/* Launch plan of one wf_step call (diagnostics). */
typedef struct {
  int32_t launches;      /* as wf_step_launch_count                                  */
  int32_t cluster;       /* CTAs (one thread-block cluster) per (sequence, head) unit */
  int32_t final_gather;  /* 1: every CTA of a unit selects the budget over all of the
                            unit's token candidates; 0: the radix select runs
                            distributed over the cluster                             */
  int32_t token_logits;  /* WF_LOGITS_*                                              */
  int32_t smem_bytes;    /* dynamic shared memory per CTA of the path kernel         */
  int32_t filter_stages; /* key tiles in flight in the filter                        */
  int32_t attend_stages; /* key/value tiles in flight in the attention               */
  int32_t stream_is_dwt_lowpass; /* two launches: 1 when the first is exactly
                            wf_dwt_lowpass (A_L only) and the second exactly the launch
                            of wf_step_cached_al on that A_L; 0 when the first also
                            forms the coarse logits the second reads (or one launch) */
  int32_t al_stages;     /* A_L stages (64 rows each) the path kernel keeps in flight
                            when it stages A_L itself (two-launch plans with
                            stream_is_dwt_lowpass = 1), else 0                       */
} wf_plan;

/* Fills *plan with the launch plan wf_step uses for these sizes on the
 * current device.  Host only; launches nothing.
 * Errors: WF_ERR_NULL/SHAPE/UNSUPPORTED, as wf_workspace_bytes. */
int wf_step_plan(const wf_dims* dims, const int32_t* k_per_level, wf_plan* plan);

/* Fault injection for tests of the bounded device waits (no counterpart in
 * the paper).  Arms a one-shot injection consumed by the next kernel launch
 * that streams K_p through mbarrier-counted bulk copies (the separate DWT
 * launch of wf_step / wf_dwt_lowpass, or the single-launch wf_step): in its
 * first CTA the first copy of the ring is never issued and the wait for it
 * gives up after `polls` polls (polls >= 1), which raises WF_DEV_WAIT_TIMEOUT
 * in the workspace status word.  Every copy that was issued is still waited
 * for, so none is in flight when the kernel ends; the launch returns WF_OK,
 * its outputs are meaningless, and later calls behave normally.
 * polls = 0 disarms.  Process-wide; not for concurrent use with other calls.
 * Errors: WF_ERR_SHAPE if polls < 0. */
int wf_debug_inject_wait_timeout(int32_t polls);

/* Clears the device status word at the start of `workspace` (async). */
int wf_clear_device_status(void* workspace, size_t workspace_bytes, void* stream);

/* Copies the device status word to *status_out and synchronises `stream`
 * (the one synchronising call of this library).  Returns WF_OK or
 * WF_ERR_CUDA; *status_out holds WF_DEV_* flags. */
int wf_read_device_status(const void* workspace, size_t workspace_bytes,
                          void* stream, int32_t* status_out);

/* Step 1 — multi-level orthonormal Haar DWT along the token axis, low-pass
 * branch only (WaveFilter §2.2 eq. (5) iterated into the pyramid of §2.2;
 * §3.1 applies it to the cached prompt keys K~[I_p]).
 *   A_j[p] = (A_{j-1}[2p] + A_{j-1}[2p+1]) / √2,  A_0 = Kp, per channel,
 * i.e. A_L[p] = 2^(-L/2) · Σ_{n = p·2^L}^{(p+1)·2^L - 1} Kp[n].
 *   Kp    : device, [U, N_p, d] of dims.dtype
 *   AL    : device, out, [U, N_p/2^L, d] fp32
 *   A_all : device, out, nullable.  If non-NULL, every level j = 1..L is
 *           written, level-major: block j holds [U, N_p/2^j, d] fp32 and
 *           blocks follow each other for j = 1, 2, ..., L.
 * Errors: WF_ERR_NULL, WF_ERR_SHAPE, WF_ERR_UNSUPPORTED, WF_ERR_ALIGNMENT,
 * WF_ERR_CUDA. */
int wf_dwt_lowpass(const wf_dims* dims, const void* Kp, float* AL, float* A_all,
                   void* stream);

/* Step 2 — importance of each coarse position and coarse Top-K (WaveFilter
 * Fig. 2(c); §1: "attention identifies the initial key tokens").
 *   z[i,p] = Q[i]·A_L[p] / √d;  s[p] = Σ_i softmax_p(z[i,·])[p];
 *   idx_L  = the k_L positions with the largest s (ties: lower p first).
 *   Q        : device, [U, G, d] of dims.dtype
 *   AL       : device, [U, N_p/2^L, d] fp32 (output of wf_dwt_lowpass)
 *   k_L      : 1 ≤ k_L ≤ N_p/2^L
 *   idx_L    : device, out, [U, k_L] int32, ascending
 *   scores_L : device, out, nullable, [U, N_p/2^L] fp32 (s)
 *   workspace: device, ≥ wf_workspace_bytes(); receives the coarse logits
 *              Q·A_L/√d of every position on the way to the scores
 * Errors: as wf_dwt_lowpass plus WF_ERR_WORKSPACE. */
int wf_score_topk(const wf_dims* dims, const void* Q, const float* AL,
                  int32_t k_L, int32_t* idx_L, float* scores_L,
                  void* workspace, size_t workspace_bytes, void* stream);

/* Step 3 — multi-scale recursive filtering down to token resolution
 * (WaveFilter Fig. 2(d); §1 "multi-scale recursive filtering").  For
 * j = L-1 .. 0: candidates C_j = {2p, 2p+1 : p ∈ S_{j+1}}, scored like
 * step 2 against A_j[C_j] (softmax over C_j), S_j = Top-k_j(C_j).
 *   Q, Kp       : device, as above (A_j is formed from the Kp rows of the
 *                 coarse survivors' spans; nothing else of Kp is read)
 *   idx_L       : device, [U, k_L] int32, the level-L survivors S_L (any
 *                 order, distinct, each in [0, N_p/2^L))
 *   k_per_level : HOST, levels+1 entries, k_per_level[j] = k_j:
 *                 k_L = entries of idx_L per unit, 1 ≤ k_j ≤ 2·k_{j+1},
 *                 k_0 = B = the final budget
 *   idx         : device, out, [U, B] int32, the token set S = S_0, ascending
 * Errors: as wf_score_topk. */
int wf_recursive_filter(const wf_dims* dims, const void* Q, const void* Kp,
                        const int32_t* idx_L, const int32_t* k_per_level,
                        int32_t* idx, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Steps 4 and 5 — gather the sparse cache and attend (WaveFilter §2.1
 * eq. (3) with the cached index set replaced by S ∪ I_g, Fig. 2(d)).
 * Keys/values are Kp/Vp rows at idx[0..B) followed by all G rows of Kg/Vg:
 *   O[i] = Σ_j softmax_j(Q[i]·K_j/√d) V_j,  lse[i] = log Σ_j exp(Q[i]·K_j/√d)
 *   idx    : device, [U, B] int32 in [0, N_p) (order free; an out-of-range
 *            entry is skipped and flagged WF_DEV_BAD_INDEX)
 *   budget : B ≥ 0 (B = 0 attends over I_g alone)
 *   O      : device, out, [U, G, d] fp32
 *   lse    : device, out, nullable, [U, G] fp32 (natural log)
 * Errors: as wf_score_topk. */
int wf_sparse_gather_attn(const wf_dims* dims, const void* Q, const void* Kp,
                          const void* Vp, const void* Kg, const void* Vg,
                          const int32_t* idx, int32_t budget, float* O,
                          float* lse, void* workspace, size_t workspace_bytes,
                          void* stream);

/* The whole per-layer, per-step path: steps 1-5 in order on `stream`.
 *   k_per_level : HOST, levels+1 entries (k_0 = budget), constraints as in
 *                 wf_recursive_filter plus 1 ≤ k_L ≤ N_p/2^L
 *   O, lse      : outputs of step 5 (lse nullable)
 *   idx_out     : device, out, nullable, [U, B] int32 — the selected tokens
 *   workspace   : device scratch of ≥ wf_workspace_bytes() bytes; holds the
 *                 coarse logits Q·A_L/√d, S_L and (for large budgets) token
 *                 logits; contents are overwritten.  Concurrent calls need
 *                 separate workspaces.
 * Errors: WF_ERR_NULL, WF_ERR_SHAPE, WF_ERR_UNSUPPORTED, WF_ERR_ALIGNMENT,
 * WF_ERR_WORKSPACE, WF_ERR_CUDA. */
int wf_step(const wf_dims* dims, const void* Q, const void* Kp, const void* Vp,
            const void* Kg, const void* Vg, const int32_t* k_per_level,
            float* O, float* lse, int32_t* idx_out, void* workspace,
            size_t workspace_bytes, void* stream);

/* wf_step reusing a level-L approximation computed at an earlier step: steps
 * 2-5 only, without the stream over K_p.  Under a prefix cache the prompt
 * keys K~[I_p] do not change between denoising steps (WaveFilter §3.1 reads
 * them at step t-1; §1 describes extracting the frequency structure with the
 * DWT at the initial step), so one wf_dwt_lowpass result serves every later
 * step of the same cache.
 *   AL : device, [U, N_p/2^L, d] fp32 — the AL output of wf_dwt_lowpass for
 *        these Kp and levels (kept by the caller; not checked).
 *   Everything else as wf_step; Kp is still read for the span rows of the
 *   coarse survivors and the selected keys.
 * Errors: as wf_step (WF_ERR_NULL if AL is NULL, WF_ERR_ALIGNMENT if it is
 * not 16-byte aligned). */
int wf_step_cached_al(const wf_dims* dims, const void* Q, const void* Kp,
                      const void* Vp, const void* Kg, const void* Vg,
                      const float* AL, const int32_t* k_per_level, float* O,
                      float* lse, int32_t* idx_out, void* workspace,
                      size_t workspace_bytes, void* stream);

/* KV-cache initialisation at the first denoising step t = 1 (WaveFilter
 * §2.1 eq. (2): the keys and values computed for every position enter the
 * cache unchanged), with the level-L approximation of the prompt keys
 * (§3.1; §1 extracts it at this initial step) written in the same pass, so
 * that later steps can call wf_step_cached_al without reading Kp for it.
 *   K, V   : device, [batch, n_prompt + n_gen, heads, head_dim] of
 *            dims.dtype, token-major (each position's heads side by side,
 *            the layout of the key/value projections' output); positions
 *            0 .. N_p-1 are the prompt I_p, N_p .. N_p+G-1 the generation
 *            block I_g
 *   Kp, Vp : device, out, [batch, heads, n_prompt, head_dim] (dims.dtype)
 *   Kg, Vg : device, out, [batch, heads, n_gen, head_dim] (dims.dtype)
 *   AL     : device, out, nullable, [U, N_p/2^L, d] fp32: A_L of Kp, the
 *            same values wf_dwt_lowpass computes (bit for bit)
 * dims: the dims of the wf_step calls that will read this cache.  Outputs
 * must not overlap the inputs.  One kernel launch.
 * Errors: WF_ERR_NULL, WF_ERR_SHAPE, WF_ERR_UNSUPPORTED, WF_ERR_ALIGNMENT,
 * WF_ERR_CUDA. */
int wf_cache_init(const wf_dims* dims, const void* K, const void* V, void* Kp,
                  void* Vp, void* Kg, void* Vg, float* AL, void* stream);

/* Cache update at a denoising step t > 1 (WaveFilter §2.1 eq. (4)): the keys
 * and values just computed for the generation positions replace the cached
 * generation rows.  The prompt rows, and an A_L computed from them, stay
 * valid.
 *   K, V   : device, [batch, n_gen, heads, head_dim] of dims.dtype,
 *            token-major
 *   Kg, Vg : device, out, [batch, heads, n_gen, head_dim]
 * dims: as for wf_step (n_prompt and levels are validated, not used).
 * Outputs must not overlap the inputs.  One kernel launch.
 * Errors: as wf_cache_init. */
int wf_cache_update(const wf_dims* dims, const void* K, const void* V, void* Kg,
                    void* Vg, void* stream);

/* Cache update over an arbitrary inferred set (WaveFilter §2.1 eq. (4),
 * K~^t[I~] = K^t[I~], V~^t[I~] = V^t[I~]): the rows of any positions — of
 * the generation block or of the prompt, as caching schemes that refresh
 * part of the prompt cache write — replace the cached ones, and the level-L
 * approximation of the prompt keys (§3.1) is re-formed at exactly the coarse
 * positions whose spans hold a rewritten prompt row (the others stay valid),
 * so wf_step_cached_al can keep running from AL without a new stream over Kp.
 *   K, V       : device, [batch, n_rows, heads, head_dim] of dims.dtype,
 *                token-major new rows
 *   positions  : device, [batch, n_rows] int32, cache positions in
 *                [0, n_prompt + n_gen) (n < n_prompt: prompt row n; else
 *                generation row n - n_prompt), distinct within a sequence
 *                (with a repeated position the row that lands is unspecified,
 *                and AL still matches the cache)
 *   Kp, Vp, Kg, Vg : device, in/out, the cache
 *   AL         : device, in/out, nullable, [U, N_p/2^L, d] fp32: A_L of Kp
 *                before the call (wf_dwt_lowpass / wf_cache_init); afterwards
 *                it equals wf_dwt_lowpass of the updated Kp bit for bit
 *   workspace  : device, nullable; if given (>= 256 bytes) a position outside
 *                the cache raises WF_DEV_BAD_INDEX in its status word (the row
 *                is skipped either way)
 * n_rows = 0 is a no-op.  Outputs must not overlap the inputs.  One or two
 * kernel launches.
 * Errors: WF_ERR_NULL, WF_ERR_SHAPE, WF_ERR_UNSUPPORTED, WF_ERR_ALIGNMENT,
 * WF_ERR_WORKSPACE, WF_ERR_CUDA. */
int wf_cache_scatter(const wf_dims* dims, const void* K, const void* V,
                     const int32_t* positions, int32_t n_rows, void* Kp, void* Vp, void* Kg,
                     void* Vg, float* AL, void* workspace, size_t workspace_bytes,
                     void* stream);

/* wf_step with host-resident inputs and outputs: copies Q/Kp/Vp/Kg/Vg from
 * HOST memory into the caller's device staging buffers (one
 * cudaMemcpyAsync each), runs wf_step, and copies O (and lse if both
 * pointers are given) back to HOST memory, all on `stream`.  Pinned host
 * memory gives asynchronous copies.  Device staging buffers d_* must have
 * the sizes of the corresponding inputs/outputs.  Does not synchronise. */
int wf_step_host(const wf_dims* dims, const void* h_Q, const void* h_Kp,
                 const void* h_Vp, const void* h_Kg, const void* h_Vg,
                 const int32_t* k_per_level, float* h_O, float* h_lse,
                 void* d_Q, void* d_Kp, void* d_Vp, void* d_Kg, void* d_Vg,
                 float* d_O, float* d_lse, void* workspace,
                 size_t workspace_bytes, void* stream);

/* One denoising step t > 1 with a device-resident cache and host-resident
 * per-step data: the serving loop that wf_cache_init (at t = 1),
 * wf_cache_update and wf_step_cached_al make possible.  On `stream`, in order:
 * copies Q and the generation block's new keys/values from HOST memory into
 * the device staging buffers (one cudaMemcpyAsync each, or a single one when
 * h_Q, h_K, h_V and d_Q, d_K, d_V each lie back to back), writes the new rows
 * into Kg/Vg (eq. (4), as wf_cache_update), runs wf_step_cached_al on the
 * cache, and copies O back to HOST memory.  Pinned host memory gives
 * asynchronous copies.  Does not synchronise.
 *   h_Q        : HOST, [batch, heads, n_gen, head_dim] (dims.dtype)
 *   h_K, h_V   : HOST, [batch, n_gen, heads, head_dim] token-major new rows
 *   h_O        : HOST, out, [batch, heads, n_gen, head_dim] fp32
 *   d_Q, d_K, d_V, d_O : device staging buffers of the same sizes
 *   Kp, Vp, AL : device, the resident prompt cache and its A_L (wf_cache_init)
 *   Kg, Vg     : device, in/out, the generation rows of the cache
 *   k_per_level, workspace : as wf_step
 * Every argument is validated before anything is enqueued.
 * Errors: as wf_step_cached_al. */
int wf_decode_step_host(const wf_dims* dims, const void* h_Q, const void* h_K,
                        const void* h_V, const int32_t* k_per_level, float* h_O,
                        void* d_Q, void* d_K, void* d_V, const void* Kp,
                        const void* Vp, void* Kg, void* Vg, const float* AL,
                        float* d_O, void* workspace, size_t workspace_bytes,
                        void* stream);

/* ---- Longer orthonormal bases (WaveFilter §3.1: the basis psi is open).
 * Readings: the basis is given by its low-pass filter g (an even number of
 * taps, 2..16, orthonormal to its even shifts); every pyramid level extends
 * its input periodically,
 *   A_j[n] = Σ_k g[k] · A_{j-1}[(2n + k) mod M],  M = N_p / 2^(j-1),
 * which keeps each level orthonormal; recursive filtering keeps the
 * pyramid's index tree (candidates at level j < L are the children 2p, 2p+1
 * of the level-(j+1) survivors) and scores them against this basis's A_j
 * exactly as the Haar path does.  With g = [1/√2, 1/√2] every result equals
 * the Haar entry points' (up to fp32 rounding order). */

/* Low-pass filter of the orthonormal Daubechies wavelet with n_moments
 * vanishing moments (1..8; 1 = Haar), extremal phase: taps_out receives
 * 2·n_moments doubles, g[0] first, summing to √2.  Host only.
 * Errors: WF_ERR_NULL, WF_ERR_UNSUPPORTED (n_moments outside 1..8). */
int wf_daubechies_lowpass(int32_t n_moments, double* taps_out);

/* Bytes of workspace wf_step_basis needs for these sizes, tap count and
 * per-level k (the route of wf_step_basis below decides: the level-L logits
 * and the path kernel's scratch, or A_1..A_L in fp32 with the candidate
 * lists, scores and logits).  Errors: as wf_workspace_bytes, plus
 * WF_ERR_UNSUPPORTED for a tap count outside 2..16 or odd. */
int wf_basis_workspace_bytes(const wf_dims* dims, int32_t taps,
                             const int32_t* k_per_level, size_t* bytes);

/* Pyramid of a longer basis: every level j = 1..L of Kp into A_all,
 * level-major ([U, N_p/2^j, d] fp32 blocks for j = 1, 2, ..., L), one launch
 * per level.  lowpass: HOST, `taps` doubles.
 * Errors: WF_ERR_NULL, WF_ERR_SHAPE, WF_ERR_UNSUPPORTED, WF_ERR_ALIGNMENT,
 * WF_ERR_CUDA. */
int wf_dwt_lowpass_basis(const wf_dims* dims, const double* lowpass,
                         int32_t taps, const void* Kp, float* A_all,
                         void* stream);

/* The whole step with a longer basis.  When every level between L and 0
 * keeps all children (k_j = 2 k_{j+1} for 0 < j < L, the default schedule),
 * the inputs are bf16, G <= 64 and the composed level-L filter has at most
 * 2048 taps ((2^L - 1)(taps - 1) + 1), two launches: the level-L logits
 * z_L[c] = Q·A_L[c]/√d with A_L[c] = Σ_m w[m] Kp[(2^L c + m) mod N_p] (the L
 * periodic levels composed into one filter w, from the taps in double), then
 * steps 2-5 of wf_step on them (the tokens under the coarse survivors are
 * the same dyadic spans for any basis and are scored on their own keys).
 * Otherwise the pyramid (L launches), the recursive filter (one CTA per
 * unit), then steps 4-5 as in wf_sparse_gather_attn.  Arguments as wf_step,
 * plus the HOST filter `lowpass` of `taps` doubles; workspace ≥
 * wf_basis_workspace_bytes() for the same sizes, taps and k.
 * Errors: as wf_step, plus WF_ERR_UNSUPPORTED for a bad tap count. */
int wf_step_basis(const wf_dims* dims, const double* lowpass, int32_t taps,
                  const void* Q, const void* Kp, const void* Vp,
                  const void* Kg, const void* Vg, const int32_t* k_per_level,
                  float* O, float* lse, int32_t* idx_out, void* workspace,
                  size_t workspace_bytes, void* stream);

/* Size of the device scratch array behind wf_step_static_scratch (48 MiB). */
#define WF_STATIC_SCRATCH_BYTES (48u << 20)

/* wf_step without a workspace argument and without any device allocation.
 * The paper has no counterpart: this entry point exists for callers that
 * cannot allocate device memory — plugin or enqueue interfaces of inference
 * engines that forbid allocation inside the call, or latency-critical loops
 * that cannot afford cudaMalloc's implicit device synchronisation.
 *   Arguments, layouts, outputs and errors: as wf_step, minus workspace.
 *   Scratch: a file-scope device array of WF_STATIC_SCRATCH_BYTES bytes that
 *   every GPU loading this library holds until the process exits.  Sizes
 *   whose wf_workspace_bytes() exceeds it are rejected with WF_ERR_WORKSPACE
 *   before anything is enqueued (e.g. the batched-long workloads at 5 % and
 *   10 % budgets).
 *   The first call on a device, with that device current, looks up the
 *   array's device address (cudaGetSymbolAddress); make that first call
 *   before any stream capture.  The address is kept for the life of the
 *   process: after cudaDeviceReset (or any other teardown of the device's
 *   primary context) this entry point must not be called again in that
 *   process.  Every call shares the one array and it keeps
 *   the last call's contents (the status word is cleared at the start of each
 *   call), so calls that overlap on the GPU — concurrent streams, or several
 *   host threads — race; serialise them.  The device status word is not
 *   readable through this entry point (use wf_step for diagnostics).
 *   Calls no cudaMalloc, cudaFree or other allocating routine. */
int wf_step_static_scratch(const wf_dims* dims, const void* Q, const void* Kp,
                           const void* Vp, const void* Kg, const void* Vg,
                           const int32_t* k_per_level, float* O, float* lse,
                           int32_t* idx_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WAVEFILTER_H_ */
