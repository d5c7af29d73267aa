/*
 * spec_verify.h - batched draft verification for speculative decoding, GB300.
 *
 * One call verifies a batch of drafted continuations against target-model
 * logits and returns, per sequence, how much of the draft is kept, the token
 * emitted where verification stops, and the buffer length to roll back to.
 *
 * Sources:
 *  - Pith review of "PipeSpec: Breaking Stage Dependencies in Hierarchical
 *    LLM Decoding" (arXiv 2505.01572), "What carries the argument": a stage
 *    verifies the previous buffer against its own prediction, appends the
 *    longest matching prefix and, on a mismatch, rolls the earlier buffers
 *    back to the last verified token.  "Circularity Check": the acceptance
 *    formula is that of Leviathan et al.  "Reading between the lines": the
 *    reported runs use greedy decoding.
 *  - "Accelerating LLM Inference with Staged Speculative Decoding"
 *    (arXiv 2308.04623), abstract: the speculative batch is a tree, and a
 *    second speculative stage is added.
 *  - Pith review of "CLaSp: In-Context Layer Skip for Self-Speculative
 *    Decoding" (arXiv 2505.24196), "Assumptions & free parameters":
 *    speculative sampling with a matching draft distribution is lossless.
 *
 * The rule (sampling mode).  p = softmax(target logits / T) and
 * q = softmax(draft logits / T) per position.  A drafted token x is kept
 * when u < min(1, p(x)/q(x)) for its uniform u in [0, 1) (strict; r >= 1
 * always keeps; q(x) = 0 keeps when p(x) > 0 and rejects when both are 0).
 * At the first rejection one token is drawn from max(0, p - q) / Z; when
 * every draft is kept one bonus token is drawn from the next target row.
 * A draw with uniform v returns the first index y (ascending) whose running
 * sum exceeds v * Z.  Greedy mode keeps a draft while it equals the target
 * argmax (ties to the lowest index) and emits the argmax where it stops;
 * greedy compares raw logits and ignores the temperature.
 *
 * Conventions for every entry point.
 *  - All array pointers are DEVICE pointers, row-major, caller-owned.  The
 *    library never allocates device memory, frees or synchronises (the one
 *    exception: spec_clasp_layer_select creates a cuBLAS handle on its first
 *    call on a device); every call is asynchronous on `stream`.  Inputs are only read; outputs are written
 *    completely (including on a data error).
 *  - Logit arrays hold float32 (SPEC_F32) or bfloat16 (SPEC_BF16) values.
 *    Row r of a logit array starts at element r * ld; only the first V
 *    elements of a row are read.  ld >= V.  Each logit array's base address
 *    must be 16-byte aligned (any ld is accepted; misaligned rows are read
 *    with realigned loads).
 *  - int arrays are int32; uniform arrays are float32 in [0, 1).
 *  - Argument errors (a NULL required pointer, a size out of range, T <= 0
 *    in sampling mode, a misaligned logit base, a short workspace) return a
 *    negative spec_status before anything is launched.  A launch failure
 *    returns SPEC_ECUDA.
 *  - Data errors found on the device never trap: they set bits in the
 *    optional per-sequence `seq_error` array and are OR-ed into the optional
 *    `*error_word` (caller zeroes it).  A sequence with bit 1, 2, 4 or 16
 *    gets empty outputs: accept length 0, tokens -1, rollback = prefix length.
 *  - Each call is two kernel launches (row statistics, then the per-sequence
 *    walk) per batch group; large sampling chain calls are split into
 *    groups that run on library streams forked from `stream` and joined
 *    back into it, so the call is ordered on `stream` like any other work.
 *    Those streams and their fork / join events belong to the calling host
 *    thread (created on its first grouped call on a device, reused after,
 *    released when the thread exits), so calls from different threads never
 *    share them; within one thread, do not enqueue a grouped call eagerly
 *    while another of the thread's calls is being captured into a graph
 *    under the global capture mode.
 *    A consulted-only chain call is one kernel (no statistics kernel);
 *    spec_compact_tree_path is one kernel; spec_clasp_layer_select is
 *    L + 2 kernels and L cuBLAS GEMMs; spec_verify_pipeline_async is one
 *    chain verification per stage and a combine kernel (see their sections).
 *  - The workspace holds the row statistics passed from the first kernel of
 *    a call to the second (8 bytes per sequence, row and 8192-element chunk).
 *    Size it with the matching *_workspace_size function; it needs no
 *    initialisation and nothing in it outlives a call.  Two calls that can
 *    run at the same time (other streams) need two workspaces.  Results are
 *    deterministic: the same inputs on the same GPU give bit-identical
 *    outputs.
 *  - Limits: B <= 65535, V <= 2,097,152.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spec_status {
  SPEC_OK = 0,
  SPEC_EINVAL = -1,      /* a size or pointer argument is invalid            */
  SPEC_EDTYPE = -2,      /* unknown dtype or mode                           */
  SPEC_EALIGN = -3,      /* a logit base address is not 16-byte aligned     */
  SPEC_EWORKSPACE = -4,  /* workspace NULL or smaller than required          */
  SPEC_ECUDA = -5        /* a CUDA launch failed                             */
} spec_status;

typedef enum spec_dtype { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;
typedef enum spec_mode { SPEC_GREEDY = 0, SPEC_SAMPLE = 1 } spec_mode;

/* data-error bits (seq_error / error_word) */
#define SPEC_ERR_TOKEN 1      /* a drafted / node token outside [0, V)          */
#define SPEC_ERR_PARENT 2     /* malformed tree parent array or depth > max     */
#define SPEC_ERR_NONFINITE 4  /* a logit row with NaN or +inf, or no finite entry */
#define SPEC_ERR_ZERO_MASS 8  /* residual mass 0 after a rejection: the token was
                                 drawn from p instead (outputs stay valid)       */
#define SPEC_ERR_INTERNAL 16  /* a bounded wait (a bulk copy of logits into shared
                                 memory, or a peer's exchange) gave up after
                                 about 65 ms; the sequence gets empty outputs
                                 (never expected; reported, not hung)          */
#define SPEC_ERR_WINDOW 32    /* asynchronous pipeline: a negative buffer length,
                                 or a stage window that does not fit in the
                                 buffer below it                                 */

/* ---------------------------------------------------------------------- */
/* Chain verification: B sequences, each with a gamma-token draft.         */
/* PipeSpec review, "What carries the argument" (longest kept prefix and   */
/* rollback); the accept / residual / bonus rule cited in its Circularity  */
/* Check.                                                                   */
/* ---------------------------------------------------------------------- */
typedef struct spec_chain_args {
  int B;                       /* sequences, >= 1                                  */
  int gamma;                   /* drafted tokens per sequence, 0..32               */
  int V;                       /* vocabulary size, >= 1                            */
  long long ld;                /* row stride of the logit arrays (elements), >= V  */
  spec_dtype dtype;
  spec_mode mode;
  float temperature;           /* > 0 and finite in SPEC_SAMPLE                     */
  const void* target_logits;   /* [B, gamma+1, ld]: row i scores position i; row
                                  gamma is the bonus position                       */
  const void* draft_logits;    /* [B, gamma, ld]; SPEC_SAMPLE only (may be NULL in
                                  greedy mode: it is not read)                      */
  const int* draft_tokens;     /* [B, gamma]                                        */
  const float* u;              /* [B, gamma] accept uniforms; SPEC_SAMPLE only      */
  const float* v;              /* [B] draw uniform; SPEC_SAMPLE only                */
  const int* prefix_len;       /* [B] tokens before the window; NULL = all 0        */
  int* accept_len;             /* out [B]: kept drafts a, 0..gamma                  */
  int* out_token;              /* out [B]: correction (a < gamma) or bonus token    */
  int* rollback_idx;           /* out [B], optional: prefix_len + a                 */
  float* p_at_draft;           /* out [B, gamma], optional: p_i(d_i) (0 in greedy)  */
  float* q_at_draft;           /* out [B, gamma], optional: q_i(d_i) (0 in greedy)  */
  float* resid_mass;           /* out [B], optional: mass Z of the distribution the
                                  token was drawn from (0 in greedy)                */
  int* seq_error;              /* out [B], optional: data-error bits                */
  int* error_word;             /* in/out, optional: data-error bits OR-ed in        */
  void* workspace;             /* 16-byte aligned, see the file comment             */
  size_t workspace_bytes;
  int consulted_only;          /* SPEC_SAMPLE only: 0 = every row is read; nonzero  */
                               /* = rows are consulted in position order (below)    */
} spec_chain_args;

/* Consulted-only mode (PipeSpec review, "What carries the argument": the  */
/* tokens after the first mismatch are rolled back unused).  One cluster   */
/* per sequence walks the positions in order and computes each position's  */
/* row statistics itself: position i's target and draft rows are read only */
/* after positions 0 .. i-1 were kept, and the bonus row only when every    */
/* draft was kept; no row after the first rejection is read.  One kernel,  */
/* no statistics kernel; the workspace is not used.  The decisions, token,  */
/* rollback and resid_mass are those of the ordinary mode; p_at_draft /     */
/* q_at_draft are NaN after the first rejection, and a NaN or +inf row is   */
/* an error only when it is read.  Greedy calls return SPEC_EINVAL in this  */
/* mode.                                                                    */
size_t spec_chain_workspace_size(int B, int gamma, int V);
spec_status spec_verify_chain(const spec_chain_args* args, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Chain verification with library-owned scratch.  None of the pages has a */
/* counterpart: this is a deployment variant of spec_verify_chain for       */
/* callers that cannot provide a workspace.  Same rule, arguments, outputs  */
/* and results as spec_verify_chain, except that args->workspace and        */
/* args->workspace_bytes are ignored: the scratch is one static device      */
/* array of SPEC_NOALLOC_SCRATCH_BYTES per device, reserved when the        */
/* library is loaded.  The call allocates and frees nothing.                */
/*  - Size limit: the call returns SPEC_EWORKSPACE, launching nothing, when */
/*    spec_chain_workspace_size(B, gamma, V) > SPEC_NOALLOC_SCRATCH_BYTES    */
/*    (e.g. B = 1024, gamma = 8, V = 131072 needs 2.2 MB and fits;          */
/*    B = 4096 at the same gamma and V needs 8.9 MB and does not).          */
/*  - The first call on a device looks up the array's device address (with  */
/*    that device current) and keeps it; make that first call before any   */
/*    stream capture.                                                       */
/*  - All calls on one device share the array: two calls that can overlap   */
/*    on the GPU (other streams, other host threads) race on it and give    */
/*    wrong results.  Serialise them, or use spec_verify_chain with one     */
/*    workspace per stream.                                                 */
/*  - The array keeps what the last call left in it.  A call reads only     */
/*    statistics it wrote itself; in consulted-only mode the control words  */
/*    that must start at zero are cleared by the call (one memset on        */
/*    `stream`).                                                            */
/* ---------------------------------------------------------------------- */
#define SPEC_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB */
spec_status spec_verify_chain_noalloc(const spec_chain_args* args, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Tree verification: each sequence carries a draft tree of N nodes.       */
/* Staged Speculative Decoding, abstract (the speculative batch as a       */
/* tree).  Row n of the logit arrays is the distribution over the children */
/* of node n; node 0 is the root (the last verified token).  Children are  */
/* tried in ascending node index.  Sampling: a child c is kept when         */
/* u[c] < min(1, p(tok_c)/q(tok_c)) for the current p; a rejected child    */
/* replaces p with max(0, p - q) renormalised (q unchanged) before the next */
/* sibling; when no child is kept the token is drawn from the current p     */
/* (from the node's own target row at a leaf).  Greedy: the first child     */
/* whose token is the target argmax is kept; otherwise the argmax is        */
/* emitted.  The walk repeats from the kept child.                          */
/* ---------------------------------------------------------------------- */
typedef struct spec_tree_args {
  int B;                       /* sequences, >= 1                                  */
  int N;                       /* nodes per tree including the root, 1..1024       */
  int max_depth;               /* deepest node allowed, 0..N-1; path_nodes has
                                  max_depth+1 entries per sequence                  */
  int V;
  long long ld;
  spec_dtype dtype;
  spec_mode mode;
  float temperature;
  const int* parent;           /* [B, N]: parent[0] = -1, 0 <= parent[i] < i      */
  const int* node_tokens;      /* [B, N]: token of node i (entry 0 not read)        */
  const void* target_logits;   /* [B, N, ld]                                        */
  const void* draft_logits;    /* [B, N, ld]; SPEC_SAMPLE only                      */
  const float* u;              /* [B, N]: u[c] for node c's own test; SPEC_SAMPLE   */
  const float* v;              /* [B]; SPEC_SAMPLE only                             */
  const int* prefix_len;       /* [B]; NULL = all 0                                 */
  int* path_len;               /* out [B]: kept nodes on the root path, 0..max_depth */
  int* path_nodes;             /* out [B, max_depth+1]: 0 (root), then the kept
                                  nodes in order, -1 padded (all -1 on a data error) */
  int* out_token;              /* out [B]                                           */
  int* rollback_idx;           /* out [B], optional: prefix_len + path_len          */
  int* seq_error;              /* out [B], optional                                 */
  int* error_word;             /* in/out, optional                                  */
  void* workspace;
  size_t workspace_bytes;
  int consulted_only;          /* 0 = every row is read; nonzero = only the rows of */
                               /* nodes the walk stands at (below)                 */
} spec_tree_args;

/* Consulted-only tree mode (Staged Speculative Decoding, abstract: the     */
/* walk keeps one child per level; PipeSpec review, "What carries the       */
/* argument": tokens after the first mismatch are never used).  One cluster */
/* per tree walks from the root and computes the statistics of node n's    */
/* rows when it stands at n: the target row always, the draft row in        */
/* sampling mode when n has children; rows of nodes off the walked path are */
/* never read.  One kernel, no statistics kernel; the workspace is not      */
/* used.  Decisions, path, token and rollback are those of the ordinary     */
/* mode on finite rows; a NaN or +inf row is an error only when it is read. */

size_t spec_tree_workspace_size(int B, int N, int V);
spec_status spec_verify_tree(const spec_tree_args* args, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* PipeSpec 3-model cascade, one synchronous snapshot: M_0 drafts O_0,     */
/* M_1 verifies it (stage 1) and M_2 verifies the first tokens of O_1      */
/* (stage 2).  PipeSpec review, "What carries the argument" and abstract;  */
/* Staged Speculative Decoding, abstract (a second speculative stage).     */
/* Stage 1: the chain rule with p = M_1, q = M_0 over the gamma1 drafts:    */
/* a1 kept, t1 = correction or bonus (M_1 row gamma1); O_1 = d[0..a1) ++ t1. */
/* Stage 2: the chain rule with p = M_2, q = M_1 over the first             */
/* w2 = min(gamma2, a1+1) tokens of O_1: a2 kept; on a rejection t2 is drawn */
/* from max(0, p2 - p1) (t2_valid = 1); when all w2 are kept no bonus is    */
/* drawn (t2 = -1, t2_valid = 0).  Rollback: a final-stage rejection rolls  */
/* O_0 back too: r0 = base0 + (rejected ? min(a1, a2) : a1),                */
/* r1 = base1 + (rejected ? a2 : w2); committed = a2 + t2_valid.            */
/* ---------------------------------------------------------------------- */
typedef struct spec_cascade_args {
  int B;
  int gamma1;                  /* stage-1 window, 1..32                             */
  int gamma2;                  /* stage-2 window, 1..min(32, gamma1+1)              */
  int V;
  long long ld;
  spec_dtype dtype;
  spec_mode mode;
  float temperature;
  const void* l0;              /* [B, gamma1, ld]   M_0 logits; SPEC_SAMPLE only    */
  const void* l1;              /* [B, gamma1+1, ld] M_1 logits                      */
  const void* l2;              /* [B, gamma2, ld]   M_2 logits                      */
  const int* draft_tokens;     /* [B, gamma1]: the O_0 window                       */
  const float* u1;             /* [B, gamma1]; SPEC_SAMPLE only                     */
  const float* v1;             /* [B]                                               */
  const float* u2;             /* [B, gamma2]                                       */
  const float* v2;             /* [B]                                               */
  const int* base0;            /* [B] length of O_0 before the window; NULL = 0     */
  const int* base1;            /* [B] length of O_1 before the window; NULL = 0     */
  int* a1;                     /* out [B] each                                      */
  int* t1;
  int* a2;
  int* w2;
  int* t2;
  int* t2_valid;
  int* r0;
  int* r1;
  int* committed;
  int* seq_error;              /* out [B], optional                                 */
  int* error_word;             /* in/out, optional                                  */
  void* workspace;
  size_t workspace_bytes;
} spec_cascade_args;

size_t spec_cascade_workspace_size(int B, int gamma1, int gamma2, int V);
spec_status spec_verify_cascade(const spec_cascade_args* args, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* k-model PipeSpec snapshot (PipeSpec review, "What carries the argument": */
/* M_0 drafts into O_0, each later M_i verifies O_{i-1} against its own      */
/* prediction and appends the verified prefix to O_i; a mismatch rolls     */
/* every earlier buffer back to the last verified token).  One synchronous  */
/* snapshot; each stage's window starts at the start of the buffer below.   */
/*  - Stage 1 is the chain rule (p = M_1, q = M_0) over the window[0]       */
/*    drafted tokens and always emits one token: the correction at the      */
/*    first rejection, else the bonus from M_1's row window[0].             */
/*  - Stage s >= 2 verifies the first w_s = min(window[s-1], len(O_{s-1}))  */
/*    tokens of O_{s-1} (p = M_s, q = M_{s-1}); it emits a correction on a   */
/*    rejection and nothing when it keeps all w_s, except the last stage     */
/*    when final_bonus is set: it then draws a bonus from M_{k-1}'s row w.   */
/*  - Rollback: buffer O_j (j = 0 .. k-2) keeps min(L_j, a_s of every        */
/*    rejecting stage s > j), L_0 = a_1, L_j = w_{j+1}; r = base + that.     */
/*  - k = 3 without the bonus is spec_verify_cascade; k = 2 is the chain.    */
/*  - Greedy mode compares argmaxes (corrections and bonus are argmaxes);   */
/*    logits[0] and the uniforms are not read.                              */
/* ---------------------------------------------------------------------- */
#define SPEC_MAX_MODELS 8
typedef struct spec_pipeline_args {
  int B;                        /* sequences, >= 1                                */
  int k;                        /* models M_0 .. M_{k-1}, 2..SPEC_MAX_MODELS      */
  int window[SPEC_MAX_MODELS - 1]; /* window[s-1]: stage s's window, 1..32        */
                                /* (window[0] = drafted tokens per sequence)       */
  int final_bonus;              /* nonzero: the last stage's bonus (see above)    */
  int V;                        /* vocabulary size, >= 1                          */
  long long ld;                 /* row stride of every logit array (elements)     */
  spec_dtype dtype;
  spec_mode mode;
  float temperature;            /* > 0 and finite in SPEC_SAMPLE                   */
  const void* logits[SPEC_MAX_MODELS];
                                /* logits[0]: M_0 [B, window[0], ld] (sampling);  */
                                /* logits[1]: M_1 [B, window[0]+1, ld];            */
                                /* logits[s], s >= 2: M_s [B, window[s-1], ld],    */
                                /* one more row for the last model with the bonus */
  const int* draft_tokens;      /* [B, window[0]]                                  */
  const float* u[SPEC_MAX_MODELS - 1]; /* u[s-1]: stage s accept uniforms        */
                                /* [B, window[s-1]] (SPEC_SAMPLE)                  */
  const float* v[SPEC_MAX_MODELS - 1]; /* v[s-1]: stage s draw uniform [B]       */
  const int* base;              /* [k-1, B] buffer lengths before the snapshot, or */
                                /* NULL (all 0)                                   */
  int* a;                       /* out [B, k-1]: tokens stage s kept              */
  int* w;                       /* out [B, k-1]: tokens stage s tested            */
  int* t;                       /* out [B, k-1]: token stage s emitted, or -1     */
  int* t_valid;                 /* out [B, k-1]: 1 when stage s emitted a token   */
  int* r;                       /* out [B, k-1]: base + kept length of O_j        */
  int* committed;               /* out [B]: len(O_{k-1})                          */
  int* seq_error;               /* out [B], optional                              */
  int* error_word;              /* in/out, optional                               */
  void* workspace;              /* 16-byte aligned, see the file comment          */
  size_t workspace_bytes;
} spec_pipeline_args;

size_t spec_pipeline_workspace_size(int B, int k, const int* window, int final_bonus, int V);
spec_status spec_verify_pipeline(const spec_pipeline_args* args, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* PipeSpec stages at independent buffer offsets: one asynchronous         */
/* snapshot.  PipeSpec review, "What carries the argument" (the models run */
/* without global synchronisation; each M_s verifies O_{s-1}, appends the  */
/* longest matching prefix, and a mismatch rolls every earlier buffer      */
/* back) and "What would settle it" (a verifier finds a full window).      */
/* Buffer O_j holds length[j][b] tokens before the snapshot.  Every stage  */
/* s = 1 .. k-1 verifies, independently of the others, the w_s tokens      */
/* O_{s-1}[l_s, l_s + w_s) with the chain rule (p = M_s, q = M_{s-1}):     */
/*  - a window must fit, l_{s-1} >= l_s + w_s (and every l_j >= 0); else   */
/*    the sequence gets SPEC_ERR_WINDOW and empty outputs;                 */
/*  - a rejection at window position a emits the correction and cuts every */
/*    earlier buffer to at most P_s = l_s + a;                             */
/*  - when every token is kept, stage 1 and (final_bonus) the last stage   */
/*    emit the bonus from M_s's row w_s, but only if position l_s + w_s is */
/*    still empty in the buffer below after that buffer's own appends in   */
/*    this snapshot (O_0 does not grow); middle stages emit nothing;       */
/*  - O_s grows to l_s + a_s (+1 when it emits); r_j = min(that, P_s over  */
/*    every rejecting stage s > j); committed = the last buffer's length.  */
/* Every stage passes w_s + 1 rows of M_s (the window's and the one after  */
/* it; the last is read even where no bonus can be emitted).  A sequence   */
/* with bit 1, 4, 16 or 32 gets empty outputs: a = 0, t = -1, t_valid = 0, */
/* r_j = l_j, committed = l_{k-1}.  Launches: one chain verification per   */
/* stage (each as spec_verify_chain), then one combine kernel.             */
/* ---------------------------------------------------------------------- */
typedef struct spec_pipeline_async_args {
  int B;                        /* sequences, 1..65535                            */
  int k;                        /* models M_0 .. M_{k-1}, 2..SPEC_MAX_MODELS      */
  int window[SPEC_MAX_MODELS - 1]; /* window[s-1] = w_s, 1..32                    */
  int final_bonus;              /* nonzero: the last stage may emit a bonus       */
  int V;                        /* vocabulary size, >= 1                          */
  long long ld;                 /* row stride of every logit array (elements)     */
  spec_dtype dtype;
  spec_mode mode;
  float temperature;            /* sampling mode, > 0                             */
  const void* target[SPEC_MAX_MODELS - 1]; /* stage s: M_s rows [B, w_s + 1]      */
  const void* draft[SPEC_MAX_MODELS - 1];  /* stage s: M_{s-1} rows [B, w_s]      */
                                /* (sampling; unused in greedy mode)               */
  const int* tokens[SPEC_MAX_MODELS - 1];  /* stage s: the window [B, w_s]        */
  const float* u[SPEC_MAX_MODELS - 1];     /* stage s: [B, w_s] (sampling)        */
  const float* v[SPEC_MAX_MODELS - 1];     /* stage s: [B] (sampling)             */
  const int* length;            /* [k, B]: l_j of sequence b at j * B + b         */
  int* a;                       /* out [B, k-1]: kept window tokens per stage     */
  int* t;                       /* out [B, k-1]: emitted token, -1 if none        */
  int* t_valid;                 /* out [B, k-1]: 1 when the stage emitted         */
  int* r;                       /* out [B, k-1]: new lengths of O_0 .. O_{k-2}    */
  int* committed;               /* out [B]: new length of O_{k-1}                 */
  int* seq_error;               /* out [B], optional                              */
  int* error_word;              /* in/out, optional                               */
  void* workspace;              /* 16-byte aligned                                */
  size_t workspace_bytes;
} spec_pipeline_async_args;

/* The largest stage's chain workspace (stages run one after another on     */
/* `stream` and share it) plus 16 bytes per (stage, sequence) of stage       */
/* results.  0 for sizes outside the limits above.                           */
size_t spec_pipeline_async_workspace_size(int B, int k, const int* window, int V);
spec_status spec_verify_pipeline_async(const spec_pipeline_async_args* args, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Cache compaction after a tree verification.  Staged Speculative         */
/* Decoding, abstract (the speculative batch is a tree); PipeSpec review,  */
/* "What carries the argument" (a buffer keeps the verified prefix and is  */
/* rolled back to the last verified token).  The verify pass wrote one row */
/* of W bytes per tree node (e.g. every layer's keys and values of that    */
/* node's token); this call copies the root's row to position prefix_len  */
/* of the sequence's contiguous cache and the i-th kept node's row to      */
/* position prefix_len + i.  No other byte of the cache changes.           */
/*  - A sequence whose path_nodes[b][0] is -1 (the verifier's data-error   */
/*    marking) is skipped and gets no error bit.                           */
/*  - A path length outside [0, max_depth], a node outside [0, N) or a     */
/*    destination past position C - 1 is a malformed path: the sequence    */
/*    is skipped (nothing written) and gets SPEC_ERR_PARENT.               */
/*  - Rows move as 16-byte vectors when W, both row strides and both base  */
/*    addresses are multiples of 16, otherwise byte by byte.               */
/*  - The tree rows and the cache must not overlap.  One kernel launch.    */
/* ---------------------------------------------------------------------- */
typedef struct spec_compact_args {
  int B;                       /* sequences, 1..65535                              */
  int N;                       /* tree nodes per sequence, >= 1                    */
  int max_depth;               /* path_nodes has max_depth + 1 columns, 0..65534  */
  int cache_rows;              /* C: cache positions per sequence, >= 1            */
  long long row_bytes;         /* W: bytes per row, >= 1                           */
  long long tree_ld;           /* bytes between consecutive node rows, >= W        */
  long long cache_ld;          /* bytes between consecutive cache positions, >= W  */
  const void* tree_rows;       /* [B][N] rows; sequence b starts at b * N * tree_ld */
  void* cache;                 /* in/out [B][C] rows; sequence b at b * C * cache_ld */
  const int* path_nodes;       /* [B, max_depth+1] (spec_verify_tree's output)     */
  const int* path_len;         /* [B] kept nodes, the root not counted             */
  const int* prefix_len;       /* [B] positions before the window; NULL = all 0    */
  int* seq_error;              /* out [B], optional: 0 or SPEC_ERR_PARENT          */
  int* error_word;             /* in/out, optional: error bits OR-ed in            */
} spec_compact_args;

spec_status spec_compact_tree_path(const spec_compact_args* args, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* CLaSp layer selection.  Pith review of "CLaSp: In-Context Layer Skip    */
/* for Self-Speculative Decoding" (arXiv 2505.24196), "What carries the    */
/* argument", and its referee report, minor comments 1 and 4.  For each    */
/* sequence, given the full model's hidden states h_0 .. h_L, choose which */
/* M of the L layers the draft skips: g(0, 0) = h_0; for i = 1 .. L and    */
/* each number of skips j, g(i, j) is the candidate with the larger cosine */
/* to h_i among f_{i-1}(g(i-1, j)) (keep layer i-1, when j <= i-1) and     */
/* g(i-1, j-1) (skip it, when j >= 1); a tie keeps the layer.  The skip    */
/* set is read back from (L, M) through the stored decisions.              */
/*  - Layer functions: f_l(x) = x + W_l x, W_l bfloat16 [d, d] row-major   */
/*    (out, in).  States are float32; the product splits x into two        */
/*    bfloat16 terms (hi = bf16(x), lo = bf16(x - hi)) and runs on the     */
/*    tensor cores with float32 accumulation, so it carries about 16       */
/*    significant bits of x.  The cosines come from float32 partial sums   */
/*    combined in double.                                                  */
/*  - Only states that can still reach (L, M) are evaluated,               */
/*    max(0, M - (L - i)) <= j <= min(i, M); others never feed g(L, M).    */
/*  - Per layer: one cuBLAS bf16 GEMM over both terms of the batch's      */
/*    states (the weights are streamed once per layer for the whole        */
/*    batch), then one DP-step kernel; an initial and a final              */
/*    (backtracking) kernel.                                               */
/*  - cuBLAS: the first call on a device creates one cuBLAS handle for the */
/*    device (cuBLAS allocates its own small state then); do not make that */
/*    first call inside a stream capture.  Calls set the handle's stream   */
/*    and point its workspace into `workspace`; calls from several host    */
/*    threads are serialised while they enqueue.                           */
/*  - Non-finite values are not checked: a NaN cosine never wins, so a     */
/*    decision involving one keeps the layer when it can.                  */
/*  - Results are deterministic for the same inputs on the same GPU.       */
/* ---------------------------------------------------------------------- */
typedef struct spec_clasp_args {
  int B;                       /* sequences, 1..65535                              */
  int L;                       /* layers, 1..4096                                  */
  int d;                       /* hidden width, a multiple of 8, 8..65536          */
  int M;                       /* layers to skip, 0..L                             */
  const float* hidden;         /* [B, L+1, d]: h_0 .. h_L; 16-byte aligned         */
  const void* weights;         /* [L, d, d] bfloat16 W_l[out][in]; 16-byte aligned */
  int* skip_mask;              /* out [B, L]: 1 where layer l is skipped, else 0   */
  float* score;                /* out [B]: D(L, M) = cos(h_L, g(L, M))             */
  unsigned char* choice;       /* out [B, L, M+1], optional: decision of state     */
                               /* (i = l+1, j) at [b, l, j]: 1 skip, 0 keep, 255   */
                               /* for states not evaluated                         */
  void* workspace;             /* 256-byte aligned, spec_clasp_workspace_size bytes */
  size_t workspace_bytes;
} spec_clasp_args;

/* Workspace for spec_clasp_layer_select: 2 (M+1) B d float32 states,        */
/* 2 (M+1) B d float32 products, 2 (M+1) B d bfloat16 split terms,           */
/* L (M+1) B decision bytes and 32 MiB for cuBLAS (each part rounded up to   */
/* 256 bytes).  0 for sizes outside the limits above.                        */
size_t spec_clasp_workspace_size(int B, int L, int d, int M);
/* SPEC_EINVAL: a size outside the limits or a NULL required pointer;        */
/* SPEC_EALIGN: hidden or weights not 16-byte aligned; SPEC_EWORKSPACE:      */
/* workspace NULL, short or not 256-byte aligned; SPEC_ECUDA: a launch or a  */
/* cuBLAS call failed (or the cuBLAS handle could not be created).           */
spec_status spec_clasp_layer_select(const spec_clasp_args* args, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Chain verification from the models' final hidden states: the LM heads    */
/* and the row statistics in one tensor-core pass.  "Accelerating LLM       */
/* Inference with Staged Speculative Decoding" (arXiv 2308.04623),         */
/* abstract: small-batch inference has low arithmetic intensity, so the    */
/* step is bound by the bytes it moves; the logits the verification reads  */
/* are what the LM head writes just before.  The rule is spec_verify_chain's.*/
/*  - Target logits at the gamma + 1 positions are H_t W_t^T, draft logits   */
/*    at the gamma positions H_d W_d^T: bfloat16 hidden states and weights,  */
/*    float32 accumulation on the tensor cores (so a logit differs from the  */
/*    exact product by float32 rounding of a d-term sum).                    */
/*  - Each head is one persistent kernel whose CTAs (or CTA pairs) own a     */
/*    slab of the vocabulary each and fold every tile of logits into per-row */
/*    (max, sum of exponentials) (sampling) or argmax (greedy) partials, the */
/*    format the chain walk merges; then the chain walk.  When the target    */
/*    head has 256 rows or more and the pairs' 256-entry tiles balance       */
/*    better than the single CTAs' tiles, both heads run on CTA pairs        */
/*    (tcgen05 cta_group::2); otherwise on one CTA per SM.                   */
/*  - Greedy mode writes no logits anywhere.  Sampling mode stores the       */
/*    float32 logits of every row in the workspace, because the residual or */
/*    bonus draw reads one or two rows per sequence chosen only after the    */
/*    accept tests; the walk reads just those rows.                          */
/*  - Same outputs, data-error bits and rules as spec_verify_chain (outputs  */
/*    as in spec_chain_args).  A bounded wait in the head kernel that gives  */
/*    up marks its rows non-finite (SPEC_ERR_NONFINITE on the affected       */
/*    sequences) and sets SPEC_ERR_INTERNAL in *error_word.                  */
/*  - Launches: one head kernel per head (the draft head only in sampling    */
/*    mode with gamma > 0), then one walk kernel.                            */
/* ---------------------------------------------------------------------- */
typedef struct spec_lm_head_chain_args {
  int B;                       /* sequences, 1..65535                              */
  int gamma;                   /* drafted tokens per sequence, 0..32               */
  int V;                       /* vocabulary size, 1..2,097,152                    */
  int d_target;                /* target hidden width, a multiple of 8, 8..65536   */
  int d_draft;                 /* draft hidden width (sampling), same limits       */
  spec_mode mode;
  float temperature;           /* > 0 and finite in SPEC_SAMPLE                     */
  const void* h_target;        /* [B, gamma+1, d_target] bfloat16, 16-byte aligned */
  const void* h_draft;         /* [B, gamma, d_draft] bfloat16 (sampling)          */
  const void* w_target;        /* [V, d_target] bfloat16 target LM head            */
  const void* w_draft;         /* [V, d_draft] bfloat16 draft LM head (sampling)   */
  const int* draft_tokens;     /* [B, gamma]                                        */
  const float* u;              /* [B, gamma] (sampling)                             */
  const float* v;              /* [B] (sampling)                                    */
  const int* prefix_len;       /* [B] or NULL                                       */
  int* accept_len;             /* out [B]                                           */
  int* out_token;              /* out [B]                                           */
  int* rollback_idx;           /* out [B], optional                                 */
  float* p_at_draft;           /* out [B, gamma], optional                          */
  float* q_at_draft;           /* out [B, gamma], optional                          */
  float* resid_mass;           /* out [B], optional                                 */
  int* seq_error;              /* out [B], optional                                 */
  int* error_word;             /* in/out, optional                                  */
  void* workspace;             /* 256-byte aligned                                  */
  size_t workspace_bytes;
} spec_lm_head_chain_args;

/* Partials: 8 bytes per (sequence, statistics row, vocabulary slab), at most */
/* 256 slabs; sampling adds the float32 logits of every row (row stride V    */
/* rounded up to a multiple of 8).  0 for sizes outside the limits.          */
size_t spec_lm_head_chain_workspace_size(int B, int gamma, int V, spec_mode mode);
/* SPEC_EINVAL: a size outside the limits or a NULL required pointer;         */
/* SPEC_EALIGN: a hidden-state or weight base not 16-byte aligned;            */
/* SPEC_EWORKSPACE: workspace NULL, short or not 256-byte aligned;            */
/* SPEC_ECUDA: a launch failed.                                               */
spec_status spec_verify_chain_lm_head(const spec_lm_head_chain_args* args, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* spec_status_string(spec_status status);

/* ---------------------------------------------------------------------- */
/* Test hook for the bounded waits (no counterpart on the pages).  While   */
/* enabled on the current device, every bulk-copy wait of a sampling      */
/* walk's residual or bonus pass (a ring stage or a resident slice) expects */
/* 16 bytes more than it copies, so it gives up after about 65 ms instead  */
/* of completing: the sequence                                             */
/* reports SPEC_ERR_INTERNAL with empty outputs and the GPU stays usable.   */
/* Nothing faults and nothing is left in flight (the copies themselves     */
/* complete).  Synchronous (one small copy to the device); affects calls   */
/* launched after it returns.  For tests of the give-up path only: leave   */
/* it disabled (the default) in any other use.                             */
/* SPEC_ECUDA if the copy fails.                                           */
/* ---------------------------------------------------------------------- */
spec_status spec_test_inject_copy_timeout(int enable);

/* ---------------------------------------------------------------------- */
/* The same kind of test hook for spec_verify_chain_lm_head.  While enabled */
/* on the current device, every pipeline stage of the head kernels (single */
/* CTAs or CTA pairs) expects 16 bytes more than it copies, so the MMA      */
/* issuers give up after about 65 ms: every row of the head comes out      */
/* non-finite (SPEC_ERR_NONFINITE on every sequence, with empty outputs)   */
/* and *error_word gets SPEC_ERR_INTERNAL.  Nothing faults and nothing is  */
/* left in flight.  Synchronous; affects calls launched after it returns.  */
/* Tests only: leave it disabled (the default) in any other use.           */
/* SPEC_ECUDA if the copy fails.                                           */
/* ---------------------------------------------------------------------- */
spec_status spec_test_inject_head_copy_timeout(int enable);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
