/* ck.h — C ABI of libck, a GB300 (sm_103a) implementation of curta-core's bit-exact
 * fixed-point transformer forward pass (phases 3 to 19), as the page "The inference core"
 * (curta.chat docs) describes it.
 *
 * Conventions
 *   - Every function returns int: 0 on success, otherwise an error number.  1 to 8 are the
 *     page's core errors (section "Core errors"); 9 and 10 are additions of this library.
 *   - Pointers named dev_* are device pointers on the current CUDA device; host_* and
 *     unqualified buffers are host memory.  `stream` is a cudaStream_t (NULL = legacy
 *     default stream).  All work is enqueued on `stream`; a call returns once its work is
 *     enqueued unless it says it synchronizes.
 *   - The library never allocates device memory for models or states: the caller allocates
 *     them (for example as torch tensors) and passes pointer and length.  The library keeps
 *     host-side handles and, per state, cached CUDA graphs.
 *   - Integer formats follow the page's table in "Fixed-point arithmetic": activations,
 *     queries, logits and scores are int64 with 16 fractional bits; cached keys and values
 *     int32 with 16; weights are bytes holding weight + 128; row scales uint32 with 24;
 *     norm weights and rotary cos/sin int32 with 24; probabilities int64 with 24; the
 *     exponential table uint32 with 30; the SiLU table int32 with 16.
 */
#ifndef CK_H
#define CK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- errors ("Core errors") */
#define CK_OK 0
#define CK_INVALID_CONFIG 1     /* a configuration value outside its range (limits below) */
#define CK_INVALID_FORMAT 2     /* an artifact that does not open with CKMODEL1 or whose
                                   directory does not fit the file or the configuration */
#define CK_INVALID_STATE 3      /* a state with the wrong tag, size, alignment, model,
                                   cursor, or one that is complete or failed */
#define CK_BUFFER_TOO_SMALL 4   /* ck_init_state given a length other than ck_state_size,
                                   or a device model buffer shorter than ck_model_size */
#define CK_MISSING_WEIGHTS 5    /* reserved: a model always holds all its matrices */
#define CK_INVALID_PROMPT 6     /* no prompt ids, an id >= vocab, max tokens 0 or above the
                                   context, or a temperature above 16 (16 << 16) */
#define CK_CONTEXT_EXCEEDED 7   /* prompt ids + max tokens - 1 above the context */
#define CK_ARITHMETIC 8         /* a key or value that does not fit the cache's 32 bits */
#define CK_CUDA_ERROR 9         /* a CUDA runtime call failed (library addition) */
#define CK_INVALID_ARGUMENT 10  /* a null pointer, misaligned pointer or size outside the
                                   documented limits (library addition) */

/* ---------------------------------------------------------------- configuration
 * Seven u32 in this order (the page: "the seven u32 values in order"; the order is the
 * llama2.c header order).  Limits of this library: every field >= 1; dim % heads == 0;
 * heads % kv_heads == 0; head size dim / heads a power of two from 4 to 128;
 * dim <= 16384; hidden <= 16384; layers <= 4095; vocab <= 1048576; context <= 32768. */
typedef struct ck_config {
  uint32_t dim, hidden, layers, heads, kv_heads, vocab, context;
} ck_config;

/* ---------------------------------------------------------------- model artifact
 * Format "CKMODEL1", little-endian; the page's artifact holds the same contents
 * ("section zero" tables and norms, matrix sections), this is the library's own layout.
 *   0   8 bytes  "CKMODEL1"
 *   8   7 x u32  ck_config
 *   36  u32      one over the square root of the head size, 24 fractional bits
 *   40  u32      flags: bit 0 = the classifier is the embedding matrix and its row scales
 *   44  u32      tensor count = 8 + 16 * layers
 *   48  u64      total artifact length in bytes
 *   56  u64      reserved (0)
 *   64  tensor directory: per tensor {u64 offset, u64 length} from the artifact start;
 *       offsets are multiples of 4; the data of a tensor is contiguous and row-major.
 * Tensors, in directory order:
 *   0 embedding       u8  [vocab][dim]       4 classifier scales u32 [vocab] (length 0 if tied)
 *   1 embedding scales u32 [vocab]           5 rotary  i32 [context][head/2][2] (cos, sin)
 *   2 final norm      i32 [dim]              6 exponential table u32 [4097]
 *   3 classifier      u8  [vocab][dim] (length 0 if tied)   7 SiLU table i32 [4097]
 *   then per layer l, at index 8 + 16 l + j:
 *   j: 0 attention norm i32[dim]  1 Wq u8[dim][dim]   2 Wq scales u32[dim]
 *      3 Wk u8[kv_dim][dim] 4 scales   5 Wv u8[kv_dim][dim] 6 scales
 *      7 Wo u8[dim][dim] 8 scales      9 feed-forward norm i32[dim]
 *      10 W1 (gate) u8[hidden][dim] 11 scales  12 W3 (up) u8[hidden][dim] 13 scales
 *      14 W2 (down) u8[dim][hidden] 15 scales
 *   with kv_dim = dim / heads * kv_heads.  Rotary pair j of a head rotates elements 2j and
 *   2j+1 of that head by entry [position][j]. */

typedef struct ck_model ck_model;

/* Validates an artifact (host memory) and reports the device bytes ck_load_model needs.
 * Errors: 2 invalid format, 1 invalid configuration, 10 null pointer. */
int ck_model_size(const void* artifact, size_t len, size_t* dev_bytes);

/* Copies an artifact into HBM in the library's kernel layout: each matrix row padded to a
 * multiple of 16 bytes; Wq, Wk, Wv stacked into one matrix; W1 and W3 rows interleaved
 * (gate row j at 2j, up row j at 2j+1).  dev_mem (256-byte aligned, dev_len >=
 * ck_model_size bytes) stays owned by the caller and must outlive the model.  The artifact
 * may be freed when the call returns (it synchronizes `stream`).
 * Errors: 1, 2, 4 (dev_len too small), 9, 10 (null or misaligned pointer). */
int ck_load_model(const void* artifact, size_t len, void* dev_mem, size_t dev_len, void* stream,
                  ck_model** out);
int ck_model_config(const ck_model* m, ck_config* out);

/* How ck_turn runs a position.  CK_PATH_STEP: one persistent kernel per position (one
 * block per SM, launched cooperatively): a producer warp streams every matrix of the
 * position through shared memory with bulk copies while consumer warps compute, with grid
 * barriers between dependent phases.  CK_PATH_KERNELS: one kernel per phase, launched with
 * programmatic dependent launch so that each kernel's weight loads start while the previous
 * one finishes.  CK_PATH_AUTO (the default) takes the phase kernels, the faster of the two on
 * every model measured; CK_PATH_STEP runs only where the model and state fit it (heads <=
 * 1000, enough shared memory and state work area).  Both compute the same bits.  Errors: 10
 * for an unknown path; ck_turn returns 10 when CK_PATH_STEP is forced on a model or state it
 * cannot run. */
#define CK_PATH_AUTO 0
#define CK_PATH_STEP 1
#define CK_PATH_KERNELS 2
int ck_set_path(ck_model* m, int path);

/* Caps the number of shared-memory ring slots (22 KB each) the one-position kernel uses;
 * 0 (the default) takes as many as fit, up to 8.  A tuning and testing control: fewer
 * slots prefetch less weight data across phase boundaries; the results are the same bits.
 * Drops the model's cached graphs.  Errors: 10 for 1 or more than 8. */
int ck_set_step_slots(ck_model* m, uint32_t max_slots);

/* The one-position kernel splits each attention head's positions over a few blocks.  Up to
 * `positions` positions (0, the default: 16384 / head dimension) every block of a head
 * scores all of them itself; beyond, the blocks score their own chunks and exchange maxima
 * and sums.  A tuning and testing control: the results are the same bits.  Drops the
 * model's cached graphs.  Errors: 10 for a null handle. */
int ck_set_attention_split(ck_model* m, uint32_t positions);

/* How far ahead of its shared-memory ring each block of the one-position kernel prefetches
 * weights into L2, in KB (0, the default: none).  Prefetches keep HBM
 * streaming while the blocks synchronise.  A tuning control: the results are the same
 * bits.  Drops the model's cached graphs.  Errors: 10 for a null handle or above 4096. */
int ck_set_step_prefetch(ck_model* m, uint32_t kb_per_block);

/* A testing control of the one-position kernel's error path: how many times each of its
 * grid and head-group barriers polls before it gives up (0, the default: about four
 * million polls, far beyond any wait a healthy position has).  A barrier that gives up
 * raises the kernel's abort word: every block stops at its next poll, its producer stops
 * issuing copies and waits for those already in flight, and the turn marks the state
 * failed and returns 9.  Waits on a block's own copies keep the default limit whatever
 * this is set to, so no copy is left in flight.  Drops the model's cached graphs.
 * Errors: 10 for a null handle. */
int ck_set_step_wait_limit(ck_model* m, uint32_t polls);

/* Layer-major prefill ("The forward pass, in order", phases 3 to 16 of prompt positions
 * that generate no token): when a turn reaches two or more such positions, ck_turn runs up
 * to `positions` of them (default 256) through each layer together, so every matrix is read
 * once per chunk and the matrix rows of the chunk are one tensor-core contraction over the
 * byte planes of the activations (exact: f16 products of 8-bit integers summed in f32 below
 * 2^24, then in 32-bit and 64-bit integers).  The state, cache and errors are the same bits
 * as position by position; a cache store that does not fit fails the state at the first
 * failing position.  The chunk's device scratch (about positions x 40 x dim bytes plus
 * 16 x positions x the widest matrix's rows) is allocated by the first such turn and kept
 * until ck_free_model or the next call.  0 or 1 turns it off.  Errors: 10 for a null
 * handle or above 4096. */
int ck_set_prefill(ck_model* m, uint32_t positions);
/* Frees the host handle, its cached CUDA graphs and its prefill scratch (not dev_mem). */
void ck_free_model(ck_model* m);

/* ---------------------------------------------------------------- state ("CKSTATE1")
 * The page's resumable state ("The resumable state") in ids mode: the run's whole
 * computation lives in one device buffer, so a state can be copied out and resumed on any
 * target (the CPU oracle reads the same layout).  Header, 256 bytes:
 *   0  "CKSTATE1"        8  u32 phase: 3 running, 20 done, 21 failed
 *   12 u32 position (the next position to run)   16 u32 prompt ids   20 u32 max tokens
 *   24 u32 cache positions = prompt ids + max tokens - 1          28 u32 generated tokens
 *   32 u32 flags (bit 0: tokens 1 and 2 complete the run)
 *   36 u32 temperature, 16 fraction bits (0: the maximum pass alone)
 *   40 u32 error (0 or 8)   44 u32 last generated token (0xFFFFFFFF before the first)
 *   48 u64 the sampling generator's state: the seed (0x9E3779B97F4A7C15 for a zero seed),
 *      advanced once per token drawn above temperature zero   56 u64 turns
 *   64 u64 first error key (all ones if none):
 *      position << 44 | layer << 32 | phase << 24 | element, phase 6 key store, 7 value
 *      store, 8 key store after rotary   72 i64 largest logit of the last generating
 *      position   80 7 x u32 the model's configuration   108 zero
 *   112 u64 sum of exponentials and 120 u64 draw of the last token sampled above temperature
 *      zero (both 0 at temperature zero)   128..255 scratch.
 * Buffers, each at a multiple of 256 bytes from the state start, in order:
 *   prompt ids u32[n_prompt], output tokens u32[max_tokens], x (activations) i64[dim],
 *   four working vectors i64[dim] (xb, q, o, y), h i64[hidden], logits i64[vocab],
 *   scores/work i64[max(heads * cache, 1024 * (head + 2) + 2048)],
 *   keys i32[layers][kv_heads][cache][head] (head-major: a head's keys for all positions are
 *   contiguous), values likewise.
 * The working vectors, h, scores/work and header bytes 128..255 are scratch: their
 * contents between turns are unspecified. */
#define CK_FLAG_STOP_TOKENS 1u
#define CK_PHASE_RUNNING 3u
#define CK_PHASE_DONE 20u
#define CK_PHASE_FAILED 21u

/* Size in bytes of a state for n_prompt ids and max_tokens.  Errors: 6, 7, 10. */
int ck_state_size(const ck_model* m, uint32_t n_prompt, uint32_t max_tokens, size_t* out);

/* The page's init_state ("The Rust API") in ids mode: zeroes the state and writes a fresh
 * header and the prompt ids (host_ids, n_ids entries, the full prompt: no opening token is
 * added).  dev_state must be 256-byte aligned and exactly ck_state_size bytes.
 * temperature_q16 (0 ..= 16 << 16, 16 fraction bits) and seed select phase 19 ("Sampling"):
 * at zero the first largest logit; above zero the sum pass over
 * EXP[min(((max - logit) / temperature) >> 8, 4096)] and a draw from xorshift64* seeded
 * with seed (a zero seed starts at 0x9E3779B97F4A7C15).
 * Errors: 3 misaligned, 4 wrong length, 6, 7, 9, 10. */
int ck_init_state(const ck_model* m, void* dev_state, size_t len, const uint32_t* host_ids,
                  uint32_t n_ids, uint32_t max_tokens, uint32_t temperature_q16, uint64_t seed,
                  uint32_t flags, void* stream);

typedef struct ck_turn_result {
  uint32_t complete;             /* the run is done or failed */
  uint32_t generated;            /* tokens generated so far */
  uint32_t generated_this_turn;
  uint32_t token;                /* last token sampled this turn, 0xFFFFFFFF if none */
  uint32_t work;                 /* positions run this turn */
  uint32_t err_position, err_layer, err_phase, err_element;  /* valid when it returns 8 */
} ck_turn_result;

/* The page's turn: runs up to n_positions positions (phases 3 to 16 per layer, and 17 to
 * 19 where a token is generated, "The forward pass, in order").  A turn is the unit of
 * host synchronisation: the call reads the state header before and after (it
 * synchronizes `stream`), and all positions in between run as CUDA-graph replays with the
 * current token kept on the device, prompt positions in layer-major chunks (see
 * ck_set_prefill).  Errors: 3 (state does not belong to the model, is
 * complete or failed, or is misaligned), 8 (a key or value did not fit 32 bits: the state
 * is marked failed, err_* name the first failing store), 9, 10. */
int ck_turn(ck_model* m, void* dev_state, size_t len, uint32_t n_positions, void* stream,
            ck_turn_result* out);

/* One position of each of n_states runs of the model, in one batched pass: the matrix rows
 * of all the runs' positions are one tensor-core contraction per matrix (the layer-major
 * kernels of ck_set_prefill), attention reads each run's own cache up to its position, and
 * each generating run samples its token (temperature and generator of its own state).  The
 * same bits as ck_turn(state, 1) on each state in turn.  dev_states: n_states distinct
 * device state pointers with their lengths in lens (host arrays); out and rcs (host arrays
 * of n_states) receive each state's turn result and return code: 0, 3 (misaligned, not
 * this model's, complete or failed: that state is left untouched), or 8 (a cache store did
 * not fit: that run is failed).  Synchronizes `stream`.  The pass's kernels run as one
 * CUDA-graph replay; the graphs (one per number of runs taking part and bound on their
 * positions, in steps of 128) are kept with the model, at most eight, and dropped by
 * ck_set_prefill and ck_free_model.  Returns the first nonzero rcs[i], else 0; 10 for null
 * arguments, repeated states or n_states of 0 or above 4096 (nothing is run), 9 for a CUDA
 * error. */
int ck_turn_batch(ck_model* m, void* const* dev_states, const size_t* lens, uint32_t n_states,
                  void* stream, ck_turn_result* out, int* rcs);

/* ck_turn_noalloc has no counterpart on the page: it exists for callers that cannot
 * allocate device memory once they are running, for example a server whose device memory
 * is carved up in advance into fixed arenas, or a host framework that owns every
 * allocation and forbids libraries from making their own.  It runs exactly one position,
 * like ck_turn with n_positions = 1 on the persistent one-position kernel, and gives the
 * same bits and the same result fields.  It allocates nothing: no cudaMalloc, no
 * cudaFree, no graph is instantiated; the kernel is launched directly.  Its scratch (the
 * grid and per-head barrier counters, attention partials and per-block classifier
 * candidates) lives in one 256 KB array in the library's device memory that every GPU
 * loading the library holds until the process exits; the state's own work region is not
 * used.  The first call on a device looks up that array's device address and sets the
 * kernel's shared-memory limit, so make it before any stream capture.  Every call shares
 * the array and clears its counters first; calls whose work overlaps on the GPU (other
 * streams, other threads) race on it and must not be issued.  Errors: those of ck_turn,
 * and 10 when the persistent kernel cannot run this model or state, or when this position
 * needs more than 256 KB of scratch.  With G blocks (the GPU's SMs, at most 768),
 * gh = G / heads blocks a head (at least 1) and P the widest padded input (dim or hidden
 * rounded up to a multiple of 128), the scratch is, each part rounded up to 256 bytes:
 * 256 + 8 * heads (cleared counters), then 16 * heads * gh + 16 * G (attention maxima and
 * sums, per-block classifier candidates), then 8 * dim (attention accumulators), then
 * 24 * P (three byte-plane buffers).  The state is still sized by ck_state_size. */
int ck_turn_noalloc(ck_model* m, void* dev_state, size_t len, void* stream, ck_turn_result* out);

/* Copies the state's logits (i64[vocab], those of the last generating position) to host
 * memory; synchronizes `stream`.  Errors: 3, 9, 10. */
int ck_logits(const ck_model* m, const void* dev_state, size_t len, int64_t* host_out,
              void* stream);

/* Phase 19 at temperature zero ("Sampling", maximum pass) over the state's logits, run as
 * a device kernel: the index of the first largest logit.  Synchronizes.  Errors: 3, 9, 10. */
int ck_argmax(const ck_model* m, const void* dev_state, size_t len, uint32_t* out, void* stream);

/* ---------------------------------------------------------------- tokenizer
 * Phases 0 to 2 ("The forward pass, in order") and the text of generated tokens
 * ("Sampling"), on the host: a prompt is tokenized once per run, before its positions.
 * The vocabulary is in llama2.c's tokenizer file layout: u32 longest token length, then per
 * token an f32 score, an i32 byte length and the bytes; token 1 opens a run, tokens 1 and 2
 * have no text, tokens 3..258 are the bytes 0..255. */
typedef struct ck_tokenizer ck_tokenizer;
/* Reads `vocab` tokens from blob (the model's vocabulary size).  Errors: 2 (the blob does
 * not hold them, or repeats a string), 10. */
int ck_tokenizer_load(const void* blob, size_t len, uint32_t vocab, ck_tokenizer** out);
void ck_tokenizer_free(ck_tokenizer* t);
/* Phases 0 to 2 on a prompt of len bytes: token 1, the token of a single space when there
 * is text, one token per UTF-8 character (or, for a character with no token, one per byte,
 * id byte + 3), then, while any adjacent pair's joined text is a token, the pair whose
 * token has the highest score merges (the leftmost of equals).  Writes the ids (*n of
 * them) for ck_init_state.  Errors: 6 (over 1,024 bytes, a zero byte, not UTF-8), 4 (cap
 * below *n), 10. */
int ck_encode(const ck_tokenizer* t, const uint8_t* text, size_t len, uint32_t* ids, uint32_t cap,
              uint32_t* n);
/* The text of ids[0..n), each after the one before it (prev before the first, e.g. the
 * last prompt id): the token's bytes, a leading space dropped right after token 1, a token
 * written <0xXX> as that one byte, nothing for tokens 1 and 2.  Writes at most cap bytes;
 * *n_bytes is the full count.  Errors: 4 (cap below *n_bytes), 10. */
int ck_decode(const ck_tokenizer* t, uint32_t prev, const uint32_t* ids, uint32_t n, uint8_t* out,
              size_t cap, size_t* n_bytes);

/* ---------------------------------------------------------------- the page's state
 * The page's resumable state ("The resumable state": CURTAST2, a 128-byte header, the
 * prompt's bytes and tokens, output tokens and text, activations, working vectors, logits,
 * scores, and the caches in [layer][position][kv_dim] order), which its core runs one chunk
 * at a time and can stop at any phase boundary, mid-layer included.  These convert between
 * it and this library's state at position boundaries (host copies of both). */
/* Size of a page state for prompt_bytes bytes of prompt and max_tokens.  Errors: 10. */
int ck_page_size(const ck_model* m, uint32_t prompt_bytes, uint32_t max_tokens, size_t* out);
/* This library's state (running or done, made with CK_FLAG_STOP_TOKENS since the page's runs
 * end at tokens 1 and 2, its prompt ids the encoding of `prompt` by t) into a page state at
 * the start of its next position (phase 3), or done (phase 20); the output text is decoded
 * with t.  Errors: 3 (not such a state), 4 (page_len not ck_page_size), 6 (prompt), 7 (the
 * page's cache would be smaller), 10. */
int ck_state_to_page(const ck_model* m, const ck_tokenizer* t, const void* host_state, size_t len,
                     const uint8_t* prompt, size_t prompt_len, void* host_page, size_t page_len);
/* A page state at a position boundary (phase 3 at layer 0, or 20) into this library's
 * state (len = ck_state_size for its prompt tokens and max tokens).  Errors: 3 (not such a
 * page state, or one stopped mid-position: run it on to the next position first), 4, 10. */
int ck_state_from_page(const ck_model* m, const void* host_page, size_t page_len, void* host_state,
                       size_t len);

/* The page's output_tokens: copies min(generated, cap) token ids to host_out and the count
 * to *n.  Synchronizes.  Errors: 3, 9, 10. */
int ck_output_tokens(const ck_model* m, const void* dev_state, size_t len, uint32_t* host_out,
                     uint32_t cap, uint32_t* n, void* stream);

/* Whole-state copies between device and host (to resume a run on another target).
 * Synchronize.  Errors: 9, 10. */
int ck_state_download(const void* dev_state, size_t len, void* host, void* stream);
int ck_state_upload(void* dev_state, const void* host, size_t len, void* stream);

/* ---------------------------------------------------------------- single matrix row kernel
 * The page's matrix row ("A matrix row") over a whole matrix on the device:
 *   sum = x[0] + ... + x[cols-1]; acc_r = sum_c byte[r][c] * x[c] (wrapping in 64 bits);
 *   y[r] = ((acc_r - 128 * sum) * scale[r]) >> 24, the multiply wrapping in 64 bits and
 *   the shift arithmetic.
 * dev_W: rows x pitch bytes, row-major, 16-byte aligned, pitch a multiple of 16 and >= cols
 * (bytes past cols are ignored); dev_scale u32[rows]; dev_x i64[cols] (8-byte aligned);
 * dev_y i64[rows].  1 <= cols <= 16384, 1 <= rows <= 2^24.  The launch allows programmatic
 * dependent launch: its weight loads may start while the previous kernel on `stream`
 * finishes, and it reads dev_x (and writes dev_y) only once that kernel has completed, so
 * stream order holds as for any launch.  Errors: 9, 10. */
int ck_matrow(const uint8_t* dev_W, size_t pitch, const uint32_t* dev_scale, uint32_t rows,
              uint32_t cols, const int64_t* dev_x, int64_t* dev_y, void* stream);

/* ---------------------------------------------------------------- host-side checks
 * Host builds of device routines, for tests without a GPU: floor square root of a u64,
 * and truncating signed division of n by d (1 <= d < 2^32) through the precomputed
 * reciprocal the normalization kernels use. */
uint64_t ck_host_isqrt(uint64_t v);
int64_t ck_host_div_trunc(int64_t n, uint32_t d);
/* A third host build: the attention probability floor((e << 24) / z) ("Attention, stage by
 * stage", stage 2) as the attention kernels form it from an estimate of 1 / z, for an
 * exponential 0 <= e <= min(z, 2^30) and a sum 2^30 <= z < 2^46. */
uint64_t ck_host_probability(uint64_t e, uint64_t z);

/* Library version string. */
const char* ck_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CK_H */
