/*
 * ciera.h -- C ABI of libciera: lossless cross-iteration exponent reuse for
 * sharded bf16 weights, on one GB300 (sm_103a).
 *
 * Method: "CIERA: Cross-Iteration Exponent Reuse for Lossless Allgather in
 * Sharded MoE Training" (Sadiq, Shen, Tanaka).  Section 3.1 (Exponent Reuse)
 * splits each bf16 value into its 8-bit exponent and a sign+mantissa byte,
 * detects per block whether any exponent changed since the previous
 * iteration, and sends only sign+mantissa for unchanged blocks; the receiver
 * rebuilds each value from its cached exponent (Appendix A, Algorithm 1).
 * Section 3.2 (Benefit-driven Selective Compression) decides per tensor
 * whether compressing pays.
 *
 * Model of the data-parallel path.  A flat buffer of N bf16 values is split
 * into R contiguous shards of S = ceil(N/R) values (the last may be short or
 * empty); rank r owns [r*S, min((r+1)*S, N)).  Each shard is cut into blocks
 * of B values (the last block of a shard may be partial).  A sender turns its
 * shard into one payload; a receiver turns all R payloads (the Allgather
 * result: rank r's payload at payloads + r*stride) back into the N values.
 *
 * Payload of one shard (len values, n_b = ceil(len/B) blocks):
 *   COMPRESSED  body || bitmap.  The body holds the blocks in order; an
 *               unchanged block contributes its len_k sign+mantissa bytes
 *               (sign in bit 7, mantissa in bits 0..6), a changed block its
 *               len_k bf16 values (2*len_k bytes, little-endian).  The bitmap
 *               has ceil(n_b/8) bytes; block k is bit (k%8) of byte k/8,
 *               padding bits are zero.
 *   RAW         the shard's 2*len bf16 bytes verbatim, no bitmap.  Chosen on
 *               a cold start, for an empty shard, or when body + bitmap would
 *               not be smaller than 2*len.  With every block changed the
 *               compressed body equals the raw bytes, so "all changed falls
 *               back to raw".
 * A block is changed iff any of its exponents differs from the sender's
 * cached exponent (an exact compare).  A cold start marks every block
 * changed.
 *
 * Conventions for every call:
 *   - Return value: CIERA_OK (0) or a negative CIERA_E_* code; no exceptions
 *     cross the ABI.  Errors found by a kernel (a corrupt descriptor on the
 *     receiver, a bounded wait that ran out) are recorded in a status word in
 *     the workspace and returned by ciera_status().
 *   - All device pointers are owned by the caller; the library allocates no
 *     device memory.  A plan owns only host metadata.
 *   - Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *     NULL means the legacy default stream).  They run on the current device.
 *   - A workspace must be zero-filled once before its first use (or passed to
 *     ciera_workspace_init) and must not be used by two calls that can run at
 *     the same time.
 *   - Fast path: when B is a multiple of 16 in [256, 16384], S is a multiple
 *     of 16, every pointer is 16-byte aligned and the payload stride is a
 *     multiple of 16, blocks are staged through shared memory with bulk
 *     copies; otherwise a byte-wise path gives the same bytes.
 */
#ifndef CIERA_H
#define CIERA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CIERA_OK 0
#define CIERA_E_INVAL (-1)       /* bad argument (size, pointer, alignment, range) */
#define CIERA_E_CUDA (-2)        /* a CUDA runtime call failed */
#define CIERA_E_CORRUPT (-3)     /* a received descriptor/bitmap does not match the plan */
#define CIERA_E_TIMEOUT (-4)     /* a bounded device-side wait ran out */
#define CIERA_E_INTERNAL (-5)    /* a kernel found its launch configuration inconsistent */
#define CIERA_E_BOUNDS (-6)      /* checked builds: an access outside its buffer was skipped */

#define CIERA_MODE_COMPRESSED 0u
#define CIERA_MODE_RAW 1u
#define CIERA_MODE_RANS 2u       /* ciera_compress_rans: exponents of changed blocks rANS-coded */

/* ciera_compress flags */
#define CIERA_COLD 1u            /* no previous exponents: every block changed, payload raw */
#define CIERA_NO_RAW_AHEAD 2u    /* every shard takes the look-back scan (no raw-ahead) */
/* ciera_decompress flags */
#define CIERA_DECOMPRESS_RANS 1u /* payloads of ciera_compress_rans: RAW or RANS */
/* Test hook: the first tile of every shard never publishes its prefix, so
 * that the tiles after it (for a raw-ahead shard: its last tile) run into
 * the bounded wait (CIERA_E_TIMEOUT). */
#define CIERA_DEBUG_SKIP_FIRST_PUBLISH 0x80000000u

typedef struct ciera_plan_s *ciera_plan_t;

/* Descriptor of one rank's payload, device-resident, 24 bytes. */
typedef struct {
    uint32_t mode;             /* CIERA_MODE_COMPRESSED, CIERA_MODE_RAW or CIERA_MODE_RANS */
    uint32_t n_changed_blocks; /* blocks whose exponents changed (all on a cold start) */
    uint64_t body_bytes;       /* bytes before the bitmap (2*len when raw) */
    uint64_t payload_bytes;    /* total bytes to send (body + bitmap, or 2*len) */
} ciera_desc;

/* Host-side facts of a plan. */
typedef struct {
    int64_t numel;             /* N */
    int64_t ranks;             /* R */
    int64_t block;             /* B */
    int64_t shard_len;         /* S = ceil(N/R) */
    int64_t blocks_per_shard;  /* ceil(S/B): per-rank stride of the flags output */
    int64_t tile_blocks;       /* blocks handled by one CTA */
    int64_t total_tiles;       /* CTAs of a full-range compress or decompress */
    int64_t payload_capacity;  /* minimum payload stride: 2*S rounded up to 256 bytes */
    int64_t workspace_bytes;   /* bytes of device workspace a call needs */
    int32_t fast_path;         /* 1 if sizes allow the shared-memory staged path */
    int32_t raw_fixup;         /* 1 if a raw payload can hold unchanged blocks (tiny B) */
} ciera_plan_info_t;

/* Cost model of the per-tensor predicate (Section 3.2, gain g_i). */
typedef struct {
    double link_Bps;           /* Allgather bandwidth the payload saves, bytes/s */
    double q_hat;              /* expected fraction of values in changed blocks */
    double t_fixed_s;          /* fixed per-tensor cost: launches, size exchange */
    double hbm_Bps;            /* receiver memory bandwidth, bytes/s */
    int64_t block;             /* block size B used for the bitmap term */
} ciera_cost_model;

/* Build a plan for a tensor of `ndim` dims `shape` (flattened, row-major),
 * block size `block` >= 1, `ranks` >= 1 simulated ranks.  Section 3.1 (block
 * partition inside each shard) and Section 3.2 (S_b = ceil(N/B)).
 * Errors: CIERA_E_INVAL for ndim < 0, a negative dim, block < 1, ranks < 1,
 * N >= 2^40, or more than 2^30 blocks per shard.  *out is set only on
 * success; free it with ciera_plan_destroy. */
int ciera_plan(const int64_t *shape, int ndim, int64_t block, int ranks, ciera_plan_t *out);

/* Fill *info.  Errors: CIERA_E_INVAL for a NULL argument. */
int ciera_plan_info(ciera_plan_t plan, ciera_plan_info_t *info);

/* Free a plan (NULL is ignored). */
void ciera_plan_destroy(ciera_plan_t plan);

/* Zero-fill a workspace of info.workspace_bytes bytes on `stream`. */
int ciera_workspace_init(ciera_plan_t plan, void *workspace_dev, void *stream);

/* Sender side (Section 3.1; Algorithm 1, sender) for ranks
 * [rank_begin, rank_begin + rank_count), all in one launch.
 *   w_dev            bf16 bit patterns of those ranks' shards, contiguous:
 *                    element 0 is the first element of shard rank_begin
 *                    (the whole tensor when rank_begin == 0 and all ranks)
 *   sender_cache_dev one exponent byte per element of the same range: the
 *                    exponents sent last iteration; updated in place
 *   payloads_dev     rank_count payload slots, slot i at
 *                    payloads_dev + i*payload_stride (>= payload_capacity)
 *   descs_dev        rank_count descriptors (device memory)
 *   flags_dev        optional (may be NULL): rank_count rows of
 *                    blocks_per_shard bytes, 1 = block changed
 *   workspace_dev    info.workspace_bytes bytes, see the conventions above
 *   flags            CIERA_COLD and/or CIERA_NO_RAW_AHEAD, or 0
 * Errors: CIERA_E_INVAL for a bad range, NULL pointer or short stride;
 * CIERA_E_CUDA if a launch fails.  CIERA_E_TIMEOUT appears later through
 * ciera_status().
 *
 * Raw-ahead.  The offsets of a compressed body depend on the changed blocks
 * of every earlier tile of the shard (the prefix scan that Algorithm 1
 * walks as "j <- j+1"), found by a look-back between the tiles' CTAs.  A
 * RAW payload needs no offsets.  A shard whose previous payload from this
 * workspace was RAW (for instance, every block of 4096 values changes each
 * step), and every shard of a cold call, is predicted RAW: its tiles store
 * their values at their raw positions without the look-back, and the
 * shard's last tile sums the tiles' changed blocks.  If the shard is not
 * RAW after all, a second kernel on the same stream rewrites its payload
 * compacted.  The bytes produced are the same either way; a wrong guess
 * costs one more read of the shard.  It applies where the staged path runs
 * (fast_path) with blocks of at least 256 values on shards of a multiple of
 * 16 values; CIERA_NO_RAW_AHEAD turns it off for a call. */
int ciera_compress(ciera_plan_t plan, int rank_begin, int rank_count, const uint16_t *w_dev,
                   uint8_t *sender_cache_dev, uint8_t *payloads_dev, int64_t payload_stride,
                   ciera_desc *descs_dev, uint8_t *flags_dev, void *workspace_dev, uint32_t flags,
                   void *stream);

/* Sender side with the paper's change test (Section 3.1; Algorithm 1,
 * "Hash128" and "HashCache"): block k is changed iff the 128-bit hash of its
 * exponents differs from hash_cache's entry for k (always on a cold start),
 * and a changed block's entry is replaced.  Same payloads, descriptors and
 * flags as ciera_compress whenever no two exponent sequences of a block
 * collide in 128 bits; the sender keeps 16 bytes per block instead of one
 * exponent byte per value, and reads 2 instead of 3 bytes per value.
 * Hash of a block of L exponents e_0..e_{L-1}, per seed s:
 *   h_s = fin(L + sum_j fin(word_j XOR splitmix64(s, j + 1)))   (mod 2^64)
 * with word_j = e_{8j} | e_{8j+1} << 8 | ... | e_{8j+7} << 56 (missing
 * exponents 0), splitmix64(s, i) the i-th output of SplitMix64 started at
 * state s, fin its output function, and seeds s1 = 0x6a09e667f3bcc908,
 * s2 = 0xbb67ae8584caa73b.
 *   hash_cache_dev  rank_count rows of blocks_per_shard entries of two
 *                   uint64 (h_s1, h_s2); updated in place
 * Other arguments as ciera_compress.  Errors: as ciera_compress, and
 * CIERA_E_INVAL when a tile holds more than 32 blocks (block < 256). */
int ciera_compress_hashed(ciera_plan_t plan, int rank_begin, int rank_count,
                          const uint16_t *w_dev, uint64_t *hash_cache_dev, uint8_t *payloads_dev,
                          int64_t payload_stride, ciera_desc *descs_dev, uint8_t *flags_dev,
                          void *workspace_dev, uint32_t flags, void *stream);

/* Sender side with the changed exponents entropy-coded (Section 3.1: the
 * sign+mantissa bytes go out as they are, the exponents that changed are
 * coded with ANS).  Change test, flags and sender cache as ciera_compress;
 * the payload of a shard of len values and n_b blocks is CIERA_MODE_RANS:
 *   [0, len)        sign+mantissa byte of every value, in order
 *   A = align16(len)                  bitmap, as in COMPRESSED payloads
 *   C = align16(A + ceil(n_b/8))      frequency table: 256 uint16, each >= 1,
 *                                     summing to 4096
 *   O = C + 512     n_b + 1 uint32: entry k = bytes of the records of the
 *                   blocks before k; entry n_b = all records' bytes
 *   D = align16(O + 4 (n_b + 1))      the records of the changed blocks
 * with zero bytes in the alignment gaps; body_bytes = D, payload_bytes = D +
 * records.  A block's record codes its L exponents with rANS (12-bit
 * probabilities, 32-bit state in [2^16, 2^32), 16-bit renormalisation) as
 * 32 interleaved lanes, lane l holding positions l, l+32, ...: 32 uint16
 * lane word counts, then each lane's words in decoding order (final state,
 * high half first, then the renormalisation words, last emitted first),
 * zero-padded to 16 bytes.  Frequencies f[s] = 1 + floor(h[s]*3840/sum h),
 * the rest of 4096 added to the most frequent symbol (lowest on a tie),
 * all 16 when h is empty, from h = hist_prev's row of the rank.  RAW as in
 * ciera_compress when cold, or when the RANS payload would not be smaller
 * than 2*len.
 *   hist_prev_dev  rank_count rows of 256 uint32: the histogram of each
 *                  shard's sampled exponents one call earlier (zeros at
 *                  first); the sample is every 16th value of the shard
 *                  (positions 0, 16, 32, ...)
 *   hist_out_dev   rank_count rows of 256 uint32, overwritten with the
 *                  histogram of this call's sampled exponents (the next
 *                  call's hist_prev); must not overlap hist_prev_dev
 * Other arguments as ciera_compress.  Errors: as ciera_compress, and
 * CIERA_E_INVAL unless the plan takes the fast path, N is a multiple of 16,
 * S <= 2^30, and w_dev, sender_cache_dev, payloads_dev (and the stride) are
 * 16-byte aligned and the histograms 4-byte aligned. */
int ciera_compress_rans(ciera_plan_t plan, int rank_begin, int rank_count, const uint16_t *w_dev,
                        uint8_t *sender_cache_dev, const uint32_t *hist_prev_dev,
                        uint32_t *hist_out_dev, uint8_t *payloads_dev, int64_t payload_stride,
                        ciera_desc *descs_dev, uint8_t *flags_dev, void *workspace_dev,
                        uint32_t flags, void *stream);

/* Receiver side (Section 3.1; Algorithm 1, receiver): rebuilds all N values
 * from the R payloads and refreshes the receiver's exponent cache.
 *   payloads_dev   R payloads, rank r's at payloads_dev + r*payload_stride
 *   descs_dev      R descriptors (device memory)
 *   recv_cache_dev N exponent bytes (ExpCache); updated in place
 *   out_dev        N bf16 outputs
 *   flags          0: payloads of ciera_compress / ciera_compress_hashed
 *                  (COMPRESSED or RAW); CIERA_DECOMPRESS_RANS: payloads of
 *                  ciera_compress_rans (RANS or RAW; a COMPRESSED payload is
 *                  then treated as corrupt), and the plan must take the fast
 *                  path, N be a multiple of 16 and every pointer be 16-byte
 *                  aligned, else CIERA_E_INVAL
 * A rank whose descriptor, bitmap or frequency table does not match the
 * plan is skipped (its output range is left untouched) and CIERA_E_CORRUPT
 * is recorded for ciera_status(); so is a RANS record that does not decode
 * cleanly (that rank's output is then undefined).  Errors: CIERA_E_INVAL,
 * CIERA_E_CUDA. */
int ciera_decompress(ciera_plan_t plan, const uint8_t *payloads_dev, int64_t payload_stride,
                     const ciera_desc *descs_dev, uint8_t *recv_cache_dev, uint16_t *out_dev,
                     void *workspace_dev, uint32_t flags, void *stream);

/* Receiver side with the R payloads in separate buffers, as a grouped
 * broadcast or any other collective that lands each rank's payload in its
 * own buffer would deliver them (Algorithm 1, receiver: one Recv() per
 * shard).  Same work and results as ciera_decompress.
 *   payload_ptrs_dev  device memory: an array of R device pointers, rank r's
 *                     payload at payload_ptrs_dev[r]; the array 8-byte aligned
 *   payload_capacity  bytes each of those buffers holds, at least
 *                     info.payload_capacity
 * Other arguments as ciera_decompress.  The pointers are read by the
 * kernels: a rank whose pointer is NULL, or (on the fast path) not 16-byte
 * aligned, is skipped like a corrupt payload and CIERA_E_CORRUPT recorded.
 * Errors: CIERA_E_INVAL (as ciera_decompress, a NULL or misaligned table, a
 * short capacity), CIERA_E_CUDA. */
int ciera_decompress_gather(ciera_plan_t plan, const uint8_t *const *payload_ptrs_dev,
                            int64_t payload_capacity, const ciera_desc *descs_dev,
                            uint8_t *recv_cache_dev, uint16_t *out_dev, void *workspace_dev,
                            uint32_t flags, void *stream);

/* One step from host memory and back: the sender side for all ranks and the
 * gather-decompress, with the weights read from host memory and the rebuilt
 * weights written to host memory (Algorithm 1 from Send to the merged
 * output), in one call.  A session owns the two copy streams and the events
 * that order them; it must not be used by two calls at once.
 *   max_chunks  the largest `chunks` a step of this session may use
 * Errors: CIERA_E_INVAL (max_chunks < 1, NULL out), CIERA_E_CUDA. */
typedef struct ciera_host_session_s *ciera_host_session_t;
int ciera_host_session_create(int max_chunks, ciera_host_session_t *out);
void ciera_host_session_destroy(ciera_host_session_t session);

/* The ranks are cut into `chunks` consecutive groups of ceil(R/chunks)
 * ranks.  For each group, in order: its values are copied from w_host into
 * w_dev on the session's upload stream; `stream` runs ciera_compress and
 * the receiver for those ranks once they have arrived; the session's
 * download stream copies the group's rebuilt values from out_dev to
 * out_host.  So the upload of one group, the kernels of the one before and
 * the download of the one before that overlap.  The step begins after the
 * work already queued on `stream` and everything it does, copies included,
 * is ordered before later work on `stream`: out_host holds the rebuilt
 * values once `stream` has been synchronised.
 *   w_host, out_host   N bf16 values in host memory; pinned (page-locked)
 *                      for the copies to run asynchronously and overlap
 *   w_dev, out_dev     N-value device buffers the call copies into / from
 *   the rest           as ciera_compress (all ranks: sender_cache_dev,
 *                      payloads_dev, payload_stride, descs_dev, flags) and
 *                      ciera_decompress (recv_cache_dev); one workspace
 *                      serves both, and ciera_status() reads its status
 *   chunks             1 .. the session's max_chunks (more than R acts as R)
 * Results equal those of ciera_compress and ciera_decompress over all ranks.
 * Errors: CIERA_E_INVAL, CIERA_E_CUDA. */
int ciera_step_host(ciera_host_session_t session, ciera_plan_t plan, const uint16_t *w_host,
                    uint16_t *out_host, uint16_t *w_dev, uint8_t *sender_cache_dev,
                    uint8_t *payloads_dev, int64_t payload_stride, ciera_desc *descs_dev,
                    uint8_t *recv_cache_dev, uint16_t *out_dev, void *workspace_dev,
                    uint32_t flags, int chunks, void *stream);

/* Wait for `stream`, then read and clear the workspace's status word.
 * Returns CIERA_OK, CIERA_E_CORRUPT, CIERA_E_TIMEOUT, CIERA_E_INTERNAL,
 * CIERA_E_BOUNDS (checked builds only) or CIERA_E_CUDA. */
int ciera_status(void *workspace_dev, void *stream);

/* Bits of a kernel status word (the status_dev output of
 * ciera_compress_noalloc; ciera_status() maps the same bits of a workspace
 * to its return codes). */
#define CIERA_STATUS_CORRUPT 1u  /* receiver: a rank did not check out (CIERA_E_CORRUPT) */
#define CIERA_STATUS_TIMEOUT 2u  /* a bounded wait ran out (CIERA_E_TIMEOUT) */
#define CIERA_STATUS_INTERNAL 4u /* inconsistent launch configuration (CIERA_E_INTERNAL) */
#define CIERA_STATUS_BOUNDS 8u   /* checked builds: an access was skipped (CIERA_E_BOUNDS) */

/* Sender side without a workspace, for callers that cannot allocate device
 * memory where they compress (inside a communication hook or an allocator
 * callback, where allocating would re-enter the allocator; or C callers with
 * no device allocator of their own).  The paper has no counterpart: this is
 * ciera_compress with the same arguments and results, except that its
 * scratch (ticket counter, status word, look-back words, flag bytes) lives
 * in a fixed 8 MiB device array inside the library, which every GPU that
 * loads the library holds until the process exits.
 *   status_dev  optional (may be NULL): one device word that receives the
 *               call's kernel status bits: 0 when its kernels finished
 *               normally, else an OR of CIERA_STATUS_TIMEOUT,
 *               CIERA_STATUS_INTERNAL and (checked builds)
 *               CIERA_STATUS_BOUNDS; the payloads of that call are then not
 *               valid
 * It allocates nothing (no cudaMalloc, no allocating library routine).  Its
 * first call on a device looks up the array's device address; make that
 * first call before any stream capture.  Every call shares the one array:
 * calls that can overlap on the GPU (other streams, other host threads)
 * race and must be serialised by the caller.  Plans of different shapes may
 * take turns: a call whose plan shape (numel, ranks, block) differs from the
 * previous call's on the device first clears the scratch it uses.
 * Errors: CIERA_E_INVAL as ciera_compress, and for a plan whose
 * info.workspace_bytes exceeds 8 MiB; CIERA_E_CUDA. */
int ciera_compress_noalloc(ciera_plan_t plan, int rank_begin, int rank_count,
                           const uint16_t *w_dev, uint8_t *sender_cache_dev, uint8_t *payloads_dev,
                           int64_t payload_stride, ciera_desc *descs_dev, uint8_t *flags_dev,
                           uint32_t *status_dev, uint32_t flags, void *stream);

/* Computation-communication pipelining on one GPU (Section 3.3): the
 * sender work of layer i+1 overlaps the receiver work of layer i.
 *
 * One layer of a step: the arguments of ciera_compress (all ranks) — or of
 * ciera_compress_rans, with `sender` = CIERA_SENDER_RANS, or of
 * ciera_compress_hashed, with `sender` = CIERA_SENDER_HASHED — and of
 * ciera_decompress for that layer's plan.  A layer's compress and
 * decompress may share one workspace; different layers must not. */
#define CIERA_SENDER_EXACT 0u
#define CIERA_SENDER_RANS 1u
#define CIERA_SENDER_HASHED 2u
typedef struct {
    ciera_plan_t plan;
    const uint16_t *w_dev;         /* all ranks' values (sender input) */
    uint8_t *sender_cache_dev;     /* exponent cache of all ranks */
    uint8_t *payloads_dev;         /* R payload slots */
    int64_t payload_stride;
    ciera_desc *descs_dev;         /* R descriptors */
    uint8_t *recv_cache_dev;       /* ExpCache, N bytes */
    uint16_t *out_dev;             /* rebuilt values, N */
    void *workspace_dev;
    uint32_t flags;                /* compress flags of this layer (CIERA_COLD, CIERA_NO_RAW_AHEAD) */
    uint32_t sender;               /* CIERA_SENDER_EXACT, _RANS or _HASHED */
    const uint32_t *hist_prev_dev; /* RANS: hist_prev of ciera_compress_rans (else unused) */
    uint32_t *hist_out_dev;        /* RANS: its hist_out */
    uint64_t *hash_cache_dev;      /* HASHED: the HashCache of ciera_compress_hashed (else
                                      unused; sender_cache_dev is then unused) */
} ciera_layer;

typedef struct ciera_pipeline_s *ciera_pipeline_t;

/* A pipeline for steps of up to max_layers layers: it owns the CUDA events
 * that order the two streams.  Errors: CIERA_E_INVAL, CIERA_E_CUDA. */
int ciera_pipeline_create(int max_layers, ciera_pipeline_t *out);
void ciera_pipeline_destroy(ciera_pipeline_t pipe);

/* Enqueue one step of n layers.  side_stream runs compress(0), compress(1),
 * ... back to back; `stream` runs decompress(i) as soon as compress(i) has
 * finished, so compress(i+1) overlaps decompress(i).  The side stream first
 * waits for everything enqueued on `stream` before the call, and `stream`'s
 * last decompress waits for all side-stream work, so the whole step is
 * ordered after earlier work on `stream` and before later work on it, and
 * can be captured into a CUDA graph from `stream` (replays then reuse the
 * captured pointers).  Results equal those of ciera_compress and
 * ciera_decompress called layer by layer.  A pipeline must not be used by
 * two calls at once.  Errors: CIERA_E_INVAL (n < 1 or > max_layers, equal
 * streams, bad layer arguments), CIERA_E_CUDA. */
int ciera_pipeline_step(ciera_pipeline_t pipe, const ciera_layer *layers, int n,
                        void *stream, void *side_stream);

/* Per-tensor predicate (Section 3.2): 1 = compress, 0 = send raw.
 * With P = N + q*N + ceil(ceil(N/B)/8) expected payload bytes,
 * compress iff (2N - P)/link_Bps > t_fixed_s + (4 + q)*N/hbm_Bps. */
int ciera_should_compress(int64_t numel);

/* Benefit-driven shard selection (Section 3.2): which of n shards to
 * compress when the receivers' exponent caches may use at most
 * cache_budget_bytes per GPU.  Shard i holds numel[i] bf16 values and has
 * block change rate q[i] in [0, 1] (measured offline).  With the process-wide
 * cost model:
 *   gain      g_i = (2 N_i - (N_i + ceil(ceil(N_i/B)/8) + q_i N_i)) / link_Bps
 *                   - (t_fixed_s + (4 + q_i) N_i / hbm_Bps)
 *   footprint M_i = (world - 1) N_i bytes (exponents of the other ranks' shards)
 * Shards with g_i > 0 are taken in descending order of g_i / M_i (equal
 * ratios: lower index first) while the total footprint fits the budget; a
 * shard that does not fit is skipped and later, smaller ones may still fit.
 * Outputs (host arrays of n): selected[i] = 1 if selected, gain[i] = g_i in
 * seconds per iteration.  The selection is made once and kept for the run.
 * Returns the number selected, or CIERA_E_INVAL (n < 0, world < 1, negative
 * budget or size, q outside [0, 1], NULL arrays with n > 0). */
int ciera_bsc_select(const int64_t *numel, const double *q, int n, int world,
                     int64_t cache_budget_bytes, uint8_t *selected, double *gain);

/* Replace / read the process-wide cost model.  Defaults: link 8e9 B/s,
 * q_hat 0.22, t_fixed 20e-6 s, hbm 8e12 B/s, block 4096.
 * Errors: CIERA_E_INVAL for NULL, non-positive rates, q_hat outside [0,1],
 * negative t_fixed or block < 1. */
int ciera_set_cost_model(const ciera_cost_model *model);
int ciera_get_cost_model(ciera_cost_model *model);

/* Limit of every bounded device-side wait, in nanoseconds (default 1 s).
 * Errors: CIERA_E_INVAL for 0. */
int ciera_set_wait_timeout_ns(uint64_t ns);

/* Static description of a status code. */
const char *ciera_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* CIERA_H */
