/*
 * ep_oracle.c -- plain, single-threaded CPU oracle for the MoE expert-parallel
 * prepare / dispatch / combine / combine_bwd / dispatch_bwd path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the package's smoke check and the benchmark's CPU-baseline
 * leg load it.  It shares no code, header, table or helper with the CUDA
 * library, and it never reads anything the CUDA path produced.
 *
 * What it computes (TransformerEngine PR #3034, "Expert Parallelism: common C
 * API + NCCL EP backend", section "Per-step (allocation-free, CUDA-graph
 * capturable)"):
 *   prepare      -- per-expert counts of the routes in topk_idx, and a routing
 *                   map whose expert blocks are padded to
 *                   dispatch_output_per_expert_alignment;
 *   dispatch     -- token rows and their routing weights placed in
 *                   expert-major receive slots;
 *   combine      -- unweighted sum of each token's expert-output rows back
 *                   in source-token order (the caller pre-multiplies);
 *   dispatch_bwd -- backward of dispatch: token and weight grads returned to
 *                   the source token;
 *   combine_bwd  -- backward of combine: the token grad copied to each of its
 *                   slots, with padded slots zeroed.
 * On one GPU all EP ranks collapse into one expert-major receive buffer, so
 * the "send" and "receive" of the pages are plain index maps here.
 *
 * Readings of points the pages leave open (each one is listed with its reason
 * in the design notes of the repository):
 *   - token_counts holds the raw per-expert route counts c_e (int32);
 *   - inside an expert block, slots follow (token, k) in ascending order;
 *   - a route of -1 is masked: no slot, contributes nothing;
 *   - an index outside [-1, E) is treated as masked and raises STATUS_BAD_INDEX;
 *   - padded rows of the receive buffers inside [0, P) are zero, P being the
 *     padded extent; rows at or beyond P are never touched;
 *   - sums are fp32, started from +0.0f, taken in ascending k, rounded once to
 *     bf16 with round-to-nearest-even;
 *   - a missing g_recv_topk_weights makes grad_topk_weights all zero;
 *   - P greater than the receive capacity R raises STATUS_OVERFLOW, and the
 *     row operations then write nothing.
 *
 * bf16 is handled as raw uint16 bit patterns; the two conversions below are
 * written from the IEEE-754 binary32 / bfloat16 layouts.
 */
#include <stdint.h>
#include <string.h>

#define STATUS_BAD_INDEX 1u
#define STATUS_OVERFLOW 2u

/* bfloat16 is the upper half of a binary32: widening appends 16 zero bits. */
float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even.  The discarded low
 * half is compared with one half ulp (0x8000): adding 0x7FFF plus the lowest
 * kept bit carries into the kept half exactly when the low half is above
 * 0x8000, or equal to it with an odd kept half.  A carry out of the mantissa
 * bumps the exponent, which is also correct (up to infinity).  NaN keeps its
 * sign and top payload bits and is made quiet. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* binary16 -> binary32 (exact): sign, 5-bit exponent (bias 15), 10-bit
 * mantissa; exponent 0 holds zero and the subnormals m * 2^-24, exponent 31
 * infinity and NaN. */
float oracle_f16_to_f32(uint16_t h) {
    uint32_t s = ((uint32_t)h & 0x8000u) << 16;
    uint32_t e = ((uint32_t)h >> 10) & 0x1Fu;
    uint32_t m = (uint32_t)h & 0x3FFu;
    uint32_t u;
    if (e == 0) {
        if (m == 0) {
            u = s;
        } else { /* subnormal: normalise m * 2^-24 */
            int shift = 0;
            while ((m & 0x400u) == 0) { m <<= 1; ++shift; }
            m &= 0x3FFu;
            u = s | ((uint32_t)(127 - 15 + 1 - shift) << 23) | (m << 13);
        }
    } else if (e == 31) {
        u = s | 0x7F800000u | (m << 13) | (m ? 0x00400000u : 0u);
    } else {
        u = s | ((e - 15 + 127) << 23) | (m << 13);
    }
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> binary16, round to nearest, ties to even.  Normal results:
 * round the 13 dropped mantissa bits like the bf16 case, then rebias the
 * exponent (a mantissa carry bumps the exponent, which is correct).  At or
 * above 65520 (halfway from 65504, the largest half, to 2^16) the result is
 * infinity.  Below 2^-14 the result is a multiple of 2^-24 rounded from the
 * full 24-bit significand; at or below 2^-25 it is zero. */
uint16_t oracle_f32_to_f16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t s = (u >> 16) & 0x8000u;
    uint32_t x = u & 0x7FFFFFFFu;
    if (x >= 0x7F800000u) return (uint16_t)(s | (x > 0x7F800000u ? 0x7E00u | ((x >> 13) & 0x3FFu) : 0x7C00u));
    if (x >= 0x477FF000u) return (uint16_t)(s | 0x7C00u);
    if (x >= 0x38800000u) {
        uint32_t r = x + 0x0FFFu + ((x >> 13) & 1u);
        r -= 0x38000000u; /* (127 - 15) << 23 */
        return (uint16_t)(s | (r >> 13));
    }
    if (x <= 0x33000000u) return (uint16_t)s;
    uint32_t e = x >> 23;                         /* 102 .. 112 */
    uint32_t m = (x & 0x7FFFFFu) | 0x800000u;     /* value = m * 2^(e-150) */
    uint32_t shift = 126u - e;                    /* to units of 2^-24 */
    uint32_t q = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (q & 1u))) q += 1u;
    return (uint16_t)(s | q);
}

/* Payload element types: 0 bf16, 1 fp16, 2 fp32. */
static float load_elem(const void* base, int64_t i, int dtype) {
    if (dtype == 0) return oracle_bf16_to_f32(((const uint16_t*)base)[i]);
    if (dtype == 1) return oracle_f16_to_f32(((const uint16_t*)base)[i]);
    return ((const float*)base)[i];
}

static void store_elem(void* base, int64_t i, int dtype, float v) {
    if (dtype == 0) ((uint16_t*)base)[i] = oracle_f32_to_bf16(v);
    else if (dtype == 1) ((uint16_t*)base)[i] = oracle_f32_to_f16(v);
    else ((float*)base)[i] = v;
}

static int64_t elem_size(int dtype) { return dtype == 2 ? 4 : 2; }

/* Step a1-a3 (prepare).  topk_idx is [T,K] row-major int64.  Outputs:
 *   token_counts[E]   c_e = number of valid routes to expert e
 *   offsets[E+1]      exclusive prefix sum of p_e = roundup(c_e, A)
 *   slot[T*K]         receive row of route (t,k), or -1 if masked/invalid
 *   inv[P]            route t*K+k held by receive row s, or -1 for padding
 *                     (caller provides room for T*K + E*(A-1) entries)
 * Returns P through *P_out and the status bits through *status_out. */
int oracle_prepare(const int64_t* topk_idx, int64_t T, int64_t K, int64_t E, int64_t A,
                   int64_t R, int32_t* token_counts, int32_t* offsets, int32_t* slot,
                   int32_t* inv, int64_t* P_out, uint32_t* status_out) {
    if (T < 0 || K < 1 || E < 1 || E > 4096 || A < 1) return -1;
    uint32_t status = 0;
    int64_t n = T * K;

    /* a1: histogram of valid routes. */
    for (int64_t e = 0; e < E; ++e) token_counts[e] = 0;
    for (int64_t r = 0; r < n; ++r) {
        int64_t e = topk_idx[r];
        if (e == -1) continue;
        if (e < -1 || e >= E) { status |= STATUS_BAD_INDEX; continue; }
        token_counts[e] += 1;
    }

    /* a2: pad each count up to a multiple of A; exclusive scan over experts. */
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) {
        int64_t c = token_counts[e];
        int64_t padded = ((c + A - 1) / A) * A;
        offsets[e + 1] = (int32_t)(offsets[e] + padded);
    }
    int64_t P = offsets[E];
    if (P > R) status |= STATUS_OVERFLOW;

    /* a3: slots in (t, k) order inside each expert block. */
    int64_t cursor[4096];
    for (int64_t e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t s = 0; s < P; ++s) inv[s] = -1;
    for (int64_t r = 0; r < n; ++r) {
        int64_t e = topk_idx[r];
        if (e < 0 || e >= E) { slot[r] = -1; continue; }
        int64_t s = cursor[e]++;
        slot[r] = (int32_t)s;
        inv[s] = (int32_t)r;
    }
    *P_out = P;
    *status_out = status;
    return 0;
}

/* Step a4 (dispatch), written per receive row: row s < P holds the token of
 * route inv[s] and that route's weight, or zeros when it is padding.  Rows
 * are H elements of the payload type, copied as bytes. */
void oracle_dispatch(const int32_t* inv, int64_t P, int64_t K, int64_t H, int dtype,
                     const void* tokens, const float* topk_weights,
                     void* recv_tokens, float* recv_topk_weights) {
    int64_t rb = H * elem_size(dtype);
    const unsigned char* src = (const unsigned char*)tokens;
    unsigned char* dst = (unsigned char*)recv_tokens;
    for (int64_t s = 0; s < P; ++s) {
        int32_t r = inv[s];
        if (r < 0) {
            for (int64_t b = 0; b < rb; ++b) dst[s * rb + b] = 0;
            recv_topk_weights[s] = 0.0f;
        } else {
            int64_t t = r / K;
            for (int64_t b = 0; b < rb; ++b) dst[s * rb + b] = src[t * rb + b];
            recv_topk_weights[s] = topk_weights[r];
        }
    }
}

/* Step a5 (combine) and the token half of a7 (dispatch_bwd): for each token,
 * the fp32 sum over k = 0..K-1 of its valid rows, rounded once to the
 * payload type (bf16 / fp16 round to nearest even; fp32 is the sum). */
void oracle_gather_sum(const int32_t* slot, int64_t T, int64_t K, int64_t H, int dtype,
                       const void* rows, void* out) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                int32_t s = slot[t * K + k];
                if (s < 0) continue;
                acc = acc + load_elem(rows, (int64_t)s * H + h, dtype);
            }
            store_elem(out, t * H + h, dtype, acc);
        }
    }
}

/* Step a6 (combine_bwd), written per receive row like dispatch: row s < P
 * gets the gradient row of the token that route inv[s] came from, or zeros. */
void oracle_combine_bwd(const int32_t* inv, int64_t P, int64_t K, int64_t H, int dtype,
                        const void* grad, void* grad_expert_out) {
    int64_t rb = H * elem_size(dtype);
    const unsigned char* src = (const unsigned char*)grad;
    unsigned char* dst = (unsigned char*)grad_expert_out;
    for (int64_t s = 0; s < P; ++s) {
        int32_t r = inv[s];
        for (int64_t b = 0; b < rb; ++b)
            dst[s * rb + b] = (r < 0) ? (unsigned char)0 : src[(int64_t)(r / K) * rb + b];
    }
}

/* Step a7, weight half: grad_topk_weights[t,k] = g_recv_topk_weights[slot],
 * zero for a masked route or when no weight gradient is given. */
void oracle_weight_gather(const int32_t* slot, int64_t T, int64_t K,
                          const float* g_recv_topk_weights, float* grad_topk_weights) {
    for (int64_t r = 0; r < T * K; ++r) {
        int32_t s = slot[r];
        grad_topk_weights[r] = (s < 0 || g_recv_topk_weights == 0) ? 0.0f : g_recv_topk_weights[s];
    }
}

/* Elementwise binary32 -> bfloat16 over an array (used to pin the rounding
 * rule against an independent implementation). */
void oracle_round_array(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}

/* Weighted combine (the optional fused weight multiply of TransformerEngine
 * PR #3035, review thread on the weight multiply in combine): each of a
 * token's rows is scaled by its receive row's routing weight in float32
 * (one rounding), the products summed in float32 from +0.0f in ascending k,
 * and the sum rounded once to bf16. */
void oracle_gather_weighted_sum(const int32_t* slot, int64_t T, int64_t K, int64_t H, int dtype,
                                const void* rows, const float* w, void* out) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                int32_t s = slot[t * K + k];
                if (s < 0) continue;
                float prod = w[s] * load_elem(rows, (int64_t)s * H + h, dtype);
                acc = acc + prod;
            }
            store_elem(out, t * H + h, dtype, acc);
        }
    }
}

/* Backward of the weighted combine, per receive row s < P holding route
 * inv[s] of token t (zeros for padding):
 *   grad_expert_out[s][h] = bf16( float32(w[s] * grad[t][h]) )
 *   g_w[s] = sum over h of grad[t][h] * expert_out[s][h]
 * The pages fix no order for the weight gradient's sum; it is returned in
 * float64 (each product of two bf16 values is exact, the sum nearly so). */
void oracle_combine_bwd_weighted(const int32_t* inv, int64_t P, int64_t K, int64_t H, int dtype,
                                 const void* grad, const float* w, const void* rows,
                                 void* grad_expert_out, double* g_w) {
    for (int64_t s = 0; s < P; ++s) {
        int32_t r = inv[s];
        if (r < 0) {
            for (int64_t h = 0; h < H; ++h) store_elem(grad_expert_out, s * H + h, dtype, 0.0f);
            g_w[s] = 0.0;
            continue;
        }
        int64_t t = r / K;
        double dot = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            float g = load_elem(grad, t * H + h, dtype);
            float prod = w[s] * g;
            store_elem(grad_expert_out, s * H + h, dtype, prod);
            dot += (double)g * (double)load_elem(rows, s * H + h, dtype);
        }
        g_w[s] = dot;
    }
}

/* Elementwise binary32 -> binary16 over an array (pinned against an
 * independent implementation). */
void oracle_round_array_f16(const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(in[i]);
}

/* Sharded prepare: expert parallelism over N ranks (TransformerEngine PR
 * #3035, "Sequence Diagram": prepare all-gathers the routing table, dispatch
 * pushes each token row to the rank that owns the chosen expert, combine
 * brings the expert rows back, and the backward pass runs the reverse
 * scatter and reverse gather).  Rank q owns the E/N experts
 * [q*E/N, (q+1)*E/N); the caller guarantees that N divides E.
 *
 * Input: every rank's topk_idx, concatenated in rank order (rank r's T_r
 * tokens follow those of ranks 0..r-1), i.e. the all-gathered table.  A route
 * is (r, t, k).  Readings: on its owner, expert e's receive block holds its
 * routes ordered by source rank, then t, then k, and is padded to a multiple
 * of A; the owner's blocks follow each other in expert order from row 0.
 * Because the concatenation lists ranks in order, "(r, t, k) ascending" is
 * plain ascending order over the concatenated routes.
 *
 * Outputs:
 *   counts[E]         valid routes per expert, over all ranks
 *   offsets[E+1]      per owner, the exclusive scan of p_e = roundup(counts[e], A)
 *                     over that owner's experts: offsets[e] is the first row of
 *                     e's block in its owner's buffer; offsets[E] = 0 is unused
 *   P[N]              rows in use on each owner (its last block's end)
 *   slot[n]           receive row of each route on its owner, or -1
 *   dest[n]           owner rank of each route, or -1
 *   inv[N * room]     per owner q, inv[q*room + s] = concatenated route index held
 *                     by row s, -1 for padding (rows at or past room are not
 *                     recorded; room = n + (E/N)*(A-1) holds every P[q])
 *   status[N]         per source rank: STATUS_BAD_INDEX for its own invalid
 *                     indices; every rank gets STATUS_OVERFLOW when some owner's
 *                     P exceeds the receive capacity R (slots are still
 *                     assigned; the row operations then write nothing). */
int oracle_shard_prepare(const int64_t* topk_idx, const int64_t* tokens_per_rank, int64_t N,
                         int64_t K, int64_t E, int64_t A, int64_t R, int64_t room,
                         int32_t* counts, int32_t* offsets, int64_t* P, int32_t* slot,
                         int32_t* dest, int32_t* inv, uint32_t* status) {
    if (N < 1 || K < 1 || E < 1 || E > 4096 || E % N != 0 || A < 1) return -1;
    int64_t Eloc = E / N;
    int64_t n = 0;
    for (int64_t q = 0; q < N; ++q) {
        if (tokens_per_rank[q] < 0) return -1;
        n += tokens_per_rank[q] * K;
        status[q] = 0;
    }
    /* the all-gathered histogram, summed over source ranks */
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    int64_t rank = 0, rank_end = tokens_per_rank[0] * K;
    for (int64_t i = 0; i < n; ++i) {
        while (i >= rank_end) { ++rank; rank_end += tokens_per_rank[rank] * K; }
        int64_t e = topk_idx[i];
        if (e == -1) continue;
        if (e < -1 || e >= E) { status[rank] |= STATUS_BAD_INDEX; continue; }
        counts[e] += 1;
    }
    /* per owner: padded blocks in expert order, starting at row 0 */
    int overflow = 0;
    for (int64_t q = 0; q < N; ++q) {
        int64_t run = 0;
        for (int64_t e = q * Eloc; e < (q + 1) * Eloc; ++e) {
            offsets[e] = (int32_t)run;
            run += ((counts[e] + A - 1) / A) * A;
        }
        P[q] = run;
        if (run > R) overflow = 1;
    }
    offsets[E] = 0;
    for (int64_t q = 0; q < N; ++q) if (overflow) status[q] |= STATUS_OVERFLOW;
    for (int64_t i = 0; i < N * room; ++i) inv[i] = -1;
    /* slots in (source rank, t, k) order inside each expert block */
    int64_t cursor[4096];
    for (int64_t e = 0; e < E; ++e) cursor[e] = offsets[e];
    for (int64_t i = 0; i < n; ++i) {
        int64_t e = topk_idx[i];
        if (e < 0 || e >= E) { slot[i] = -1; dest[i] = -1; continue; }
        int64_t q = e / Eloc;
        int64_t s = cursor[e]++;
        slot[i] = (int32_t)s;
        dest[i] = (int32_t)q;
        if (s < room) inv[q * room + s] = (int32_t)i;
    }
    return 0;
}

/* Sharded combine (token half of the sharded dispatch_bwd too): route i of
 * the concatenated table reads row slot[i] of its owner dest[i]'s buffer,
 * rows_of_rank[dest[i]]; per token the float32 sum over k from +0.0f in
 * ascending k, rounded once to the payload type -- the single-buffer sum
 * with each row fetched from its owner. */
void oracle_shard_gather_sum(const int32_t* slot, const int32_t* dest, int64_t T, int64_t K,
                             int64_t H, int dtype, const void* const* rows_of_rank, void* out) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int64_t k = 0; k < K; ++k) {
                int32_t s = slot[t * K + k];
                if (s < 0) continue;
                acc = acc + load_elem(rows_of_rank[dest[t * K + k]], (int64_t)s * H + h, dtype);
            }
            store_elem(out, t * H + h, dtype, acc);
        }
    }
}

/* Sharded dispatch_bwd, weight half: grad_topk_weights[i] = the weight
 * gradient of route i's receive row on its owner, 0 for a masked route or
 * when no weight gradient is given (g_of_rank == 0). */
void oracle_shard_weight_gather(const int32_t* slot, const int32_t* dest, int64_t n,
                                const float* const* g_of_rank, float* grad_topk_weights) {
    for (int64_t i = 0; i < n; ++i) {
        int32_t s = slot[i];
        grad_topk_weights[i] = (s < 0 || g_of_rank == 0) ? 0.0f : g_of_rank[dest[i]][s];
    }
}

/* ----------------------------------------------------------------------------
 * Rank-major receive layout (TransformerEngine PR #3035, review thread on the
 * receive buffers: a rank-major buffer needs max_tokens_per_rank x num_ranks
 * rows at worst, the expert-major one that times min(topk, E); the owner then
 * permutes the received rows locally into expert-major order).
 *
 * Readings (the thread names the layout, not its details):
 *   - a token goes once to every rank that owns at least one of its valid
 *     routes (rank q owns experts [q*E/N, (q+1)*E/N));
 *   - owner q's buffer lists, source ranks in order, each rank's tokens that
 *     go to q, tokens ascending, with no gap between source blocks;
 *   - with each row go the token's K expert ids relative to q (-1 where the
 *     route is masked, invalid or owned by another rank) and its K routing
 *     weights (0.0f there): the input of the owner's local single-buffer
 *     prepare and dispatch, which do the permutation;
 *   - combine sums, per token, the owners' partial rows (each already the
 *     owner's local combine) in the order in which each owner first appears
 *     among the token's routes, k ascending, in float32 from +0.0f, rounded
 *     once; the backward passes mirror this.
 *
 * Inputs are the ranks' topk_idx tables concatenated in rank order, as in
 * oracle_shard_prepare.  Outputs:
 *   counts[N*N]      counts[r*N + q] = tokens of rank r that go to owner q
 *   M[N]             rows each owner receives (sum over r of counts[r*N + q])
 *   row[n]           for every valid route, the row of its token on the
 *                    route's owner (repeated owners share the row); -1 else
 *   dest[n]          the owner of every valid route; -1 else
 *   first[n]         1 where the route is its owner's first in the token
 *   src[N*room]      per owner q, src[q*room + s] = concatenated token index
 *                    held by row s (rows at or past room are not recorded;
 *                    room = total tokens holds every M[q])
 *   status[N]        STATUS_BAD_INDEX for a rank's own invalid indices; every
 *                    rank gets STATUS_OVERFLOW when some M[q] exceeds R. */
int oracle_rm_prepare(const int64_t* topk_idx, const int64_t* tokens_per_rank, int64_t N,
                      int64_t K, int64_t E, int64_t R, int64_t room, int32_t* counts, int64_t* M,
                      int32_t* row, int32_t* dest, int32_t* first, int64_t* src, uint32_t* status) {
    if (N < 1 || N > 64 || K < 1 || E < 1 || E % N != 0) return -1;
    int64_t Eloc = E / N;
    int64_t T = 0;
    for (int64_t r = 0; r < N; ++r) {
        if (tokens_per_rank[r] < 0) return -1;
        T += tokens_per_rank[r];
        status[r] = 0;
    }
    if (room < T) return -1;
    for (int64_t i = 0; i < N * N; ++i) counts[i] = 0;
    for (int64_t i = 0; i < N * room; ++i) src[i] = -1;
    /* pass 1: per token, which owners it goes to; counts per (source, owner) */
    int64_t rank = 0, rank_end = tokens_per_rank[0];
    for (int64_t g = 0; g < T; ++g) {
        while (g >= rank_end) { ++rank; rank_end += tokens_per_rank[rank]; }
        int goes[64];
        for (int64_t q = 0; q < N; ++q) goes[q] = 0;
        for (int64_t k = 0; k < K; ++k) {
            int64_t e = topk_idx[g * K + k];
            if (e < -1 || e >= E) status[rank] |= STATUS_BAD_INDEX;
            if (e < 0 || e >= E) continue;
            goes[e / Eloc] = 1;
        }
        for (int64_t q = 0; q < N; ++q) counts[rank * N + q] += goes[q];
    }
    int overflow = 0;
    for (int64_t q = 0; q < N; ++q) {
        M[q] = 0;
        for (int64_t r = 0; r < N; ++r) M[q] += counts[r * N + q];
        if (M[q] > R) overflow = 1;
    }
    for (int64_t r = 0; r < N; ++r) if (overflow) status[r] |= STATUS_OVERFLOW;
    /* pass 2: rows in (source rank, token) order on each owner; because the
     * concatenation lists ranks in order, that is plain token order */
    int64_t cursor[64];
    for (int64_t q = 0; q < N; ++q) cursor[q] = 0;
    for (int64_t g = 0; g < T; ++g) {
        int64_t row_of[64];
        for (int64_t q = 0; q < N; ++q) row_of[q] = -1;
        for (int64_t k = 0; k < K; ++k) {
            int64_t i = g * K + k, e = topk_idx[i];
            if (e < 0 || e >= E) { row[i] = -1; dest[i] = -1; first[i] = 0; continue; }
            int64_t q = e / Eloc;
            first[i] = row_of[q] < 0;
            if (row_of[q] < 0) {
                row_of[q] = cursor[q]++;
                if (row_of[q] < room) src[q * room + row_of[q]] = g;
            }
            row[i] = (int32_t)row_of[q];
            dest[i] = (int32_t)q;
        }
    }
    return 0;
}

/* Rank-major dispatch on owner q: row s of its buffer is the token
 * tokens[src[s]], with that token's K ids relative to q (-1 for routes q does
 * not own) and their weights (0.0f there).  weights may be 0 (ids and rows
 * only). */
void oracle_rm_dispatch(const int64_t* src, int64_t M, const int64_t* topk_idx,
                        const float* topk_weights, int64_t K, int64_t E, int64_t N, int64_t q,
                        int64_t H, int dtype, const void* tokens, void* recv_tokens,
                        int64_t* recv_idx, float* recv_weights) {
    int64_t Eloc = E / N, es = elem_size(dtype);
    for (int64_t s = 0; s < M; ++s) {
        int64_t g = src[s];
        memcpy((char*)recv_tokens + s * H * es, (const char*)tokens + g * H * es, (size_t)(H * es));
        for (int64_t k = 0; k < K; ++k) {
            int64_t e = topk_idx[g * K + k];
            int mine = e >= 0 && e < E && e / Eloc == q;
            recv_idx[s * K + k] = mine ? e - q * Eloc : -1;
            if (recv_weights) recv_weights[s * K + k] = mine && topk_weights ? topk_weights[g * K + k] : 0.0f;
        }
    }
}

/* Rank-major dispatch_bwd, weight half: grad_topk_weights[g*K + k] = owner
 * dest's weight gradient for its row of token g, entry k; 0 for a masked
 * route or when no weight gradients are given (g_of_rank == 0). */
void oracle_rm_weight_gather(const int32_t* row, const int32_t* dest, int64_t T, int64_t K,
                             const float* const* g_of_rank, float* grad_topk_weights) {
    for (int64_t g = 0; g < T; ++g)
        for (int64_t k = 0; k < K; ++k) {
            int64_t i = g * K + k;
            grad_topk_weights[i] = (row[i] < 0 || g_of_rank == 0)
                                       ? 0.0f : g_of_rank[dest[i]][(int64_t)row[i] * K + k];
        }
}
