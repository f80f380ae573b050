// prefill_generic.cu -- chunkwise WY/UT prefill on CUDA cores, float32.
//
// Page "Reorder channelwise gated delta rule chunked hot loops for
// autovectorization" (pytorch/executorch PR #21021), second commit summary:
// for T != 1 the forward runs chunk by chunk, computing per-channel
// log-decay prefixes, causal query/key terms, a beta-folded triangular
// transform, WY pseudo-keys and pseudo-values, and the state carried from one
// chunk to the next; a ragged last chunk goes through the same code.
//
// The algebra (unrolling the per-token recurrence over one chunk of L tokens,
// local indices r, s; S0 = state at the chunk start; G = inclusive prefix sum
// of g over the chunk per key channel):
//   A[r,s] = beta_r sum_i k_ri k_si exp(G_ri - G_si)      s <  r  (else 0)
//   P[r,s] =        sum_i q_ri k_si exp(G_ri - G_si)      s <= r  (else 0)
//   Wk = (I + A)^-1 diag(beta) (exp(G) * K)    WY pseudo-keys    [L, dk]
//   Wv = (I + A)^-1 diag(beta) V               WY pseudo-values  [L, dv]
//   U  = Wv - Wk S0
//   O  = (exp(G) * Q) S0 + P U
//   S  = diag(exp(G_L)) S0 + (exp(G_L - G) * K)^T U
// Every exponent used is <= 0 (the decay between two tokens, taken in causal
// order), so nothing overflows whatever the strength of the decay.
//
// This is the general path: any supported (dk, dv, chunk) and both dtypes,
// float32 throughout, with exact pairwise decays.  Two kernels:
//   gdr_chunk_prep  one CTA per (batch, value head, chunk), all chunks in
//                   parallel: prefix sums, A and P, the unit-lower solve by
//                   forward substitution, and the per-chunk operands of the
//                   scan, written to the workspace;
//   gdr_chunk_scan  one CTA per (batch, value head, 32-column tile of dv),
//                   sequential over chunks: U, O and the state carry, with
//                   the state tile resident in shared memory.
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace gdr {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kScanThreads = 256;
constexpr int kScanBV = 32;

// Per (b, hv, chunk) workspace record, in floats:
//   Wk [C][dk] | Qt [C][dk] | Kh [C][dk] | Wv [C][dv] | P [C][C] | gam [dk]
struct ChunkLayout {
    int C, dk, dv;
    __host__ __device__ size_t wk() const { return 0; }
    __host__ __device__ size_t qt() const { return (size_t)C * dk; }
    __host__ __device__ size_t kh() const { return 2 * (size_t)C * dk; }
    __host__ __device__ size_t wv() const { return 3 * (size_t)C * dk; }
    __host__ __device__ size_t p() const { return 3 * (size_t)C * dk + (size_t)C * dv; }
    __host__ __device__ size_t gam() const { return p() + (size_t)C * C; }
    __host__ __device__ size_t floats() const {
        // keep each record a multiple of 4 floats (16 bytes)
        return (gam() + dk + 3) & ~(size_t)3;
    }
};

// ---- 3xTF32 warp products: an f32 x is split exactly into a
// tf32 head (x with its 13 low mantissa bits cleared) and the f32 rest
// x - head; a product is head*head + head*rest + rest*head, the rest*rest
// term (~2^-22 relative) dropped, and the tensor core reads the rest's top
// 19 bits.  m16n8k8 fragments (g = lane / 4, t = lane % 4): A holds
// (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4); B (t, g), (t + 4, g); the
// accumulator (g, 2t), (g, 2t + 1), (g + 8, 2t), (g + 8, 2t + 1).
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    hi = __float_as_uint(x) & 0xffffe000u;
    lo = __float_as_uint(x - __uint_as_float(hi));
}

__device__ __forceinline__ void mma_tf32_acc(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte asynchronous copy global -> shared (L2 only), and the wait for all
// of this thread's copies.
__device__ __forceinline__ void cp_async16(float *dst, const float *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all_copies() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// The split A fragment of a 16 x 8 block at (m0, k0): element (row, col) at
// A[row * lda + col] (or, TRANS_A, at A[col * lda + row]), times sign.
template <bool TRANS_A>
__device__ __forceinline__ void load_a3(uint32_t (&ah)[4], uint32_t (&al)[4], const float *A,
                                        int lda, int m0, int k0, float sign, int g, int t) {
    auto a_at = [&](int r, int c) {
        return TRANS_A ? A[(k0 + c) * lda + m0 + r] : A[(m0 + r) * lda + k0 + c];
    };
    split_tf32(sign * a_at(g, t), ah[0], al[0]);
    split_tf32(sign * a_at(g + 8, t), ah[1], al[1]);
    split_tf32(sign * a_at(g, t + 4), ah[2], al[2]);
    split_tf32(sign * a_at(g + 8, t + 4), ah[3], al[3]);
}

// acc (16 x 8) += A B for one k-step of 8 with a split A fragment; B element
// (k, n) at B[k * ldb + n] (or, TRANS_B, at B[n * ldb + k]).
template <bool TRANS_B>
__device__ __forceinline__ void mma3_b(float (&acc)[4], const uint32_t (&ah)[4],
                                       const uint32_t (&al)[4], const float *B, int ldb, int k0,
                                       int n0, int g, int t) {
    auto b_at = [&](int k, int n) {
        return TRANS_B ? B[(n0 + n) * ldb + k0 + k] : B[(k0 + k) * ldb + n0 + n];
    };
    uint32_t bh0, bl0, bh1, bl1;
    split_tf32(b_at(t, g), bh0, bl0);
    split_tf32(b_at(t + 4, g), bh1, bl1);
    mma_tf32_acc(acc, al, bh0, bh1);
    mma_tf32_acc(acc, ah, bl0, bl1);
    mma_tf32_acc(acc, ah, bh0, bh1);
}

// NT adjacent 16 x 8 tiles of one row block: acc[n] += sign * A[m0.., 0..kend)
// B[0..kend, nbase + 8 n ..].  k runs outermost, so the A fragment is split
// once per k-step for all NT tiles, and the head*head products and the two
// correction products go to separate accumulators: 2 NT independent chains
// instead of one per tile.
template <int NT, bool TRANS_A>
__device__ __forceinline__ void mma3_rows(float (&acc)[NT][4], const float *A, int lda, int m0,
                                          int kend, const float *B, int ldb, int nbase,
                                          float sign, int g, int t) {
    float cor[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) cor[n][0] = cor[n][1] = cor[n][2] = cor[n][3] = 0.f;
    for (int k0 = 0; k0 < kend; k0 += 8) {
        uint32_t ah[4], al[4];
        load_a3<TRANS_A>(ah, al, A, lda, m0, k0, sign, g, t);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            uint32_t bh0, bl0, bh1, bl1;
            split_tf32(B[(k0 + t) * ldb + nbase + 8 * n + g], bh0, bl0);
            split_tf32(B[(k0 + t + 4) * ldb + nbase + 8 * n + g], bh1, bl1);
            mma_tf32_acc(cor[n], al, bh0, bh1);
            mma_tf32_acc(cor[n], ah, bl0, bl1);
            mma_tf32_acc(acc[n], ah, bh0, bh1);
        }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] += cor[n][e];
}


// TREE: the T <= C tokens of each (b, hv) are a draft-token tree given by
// parents[b][t] (-1 for a root, else an earlier token), solved as one chunk:
// prefix sums run along root paths and the ancestor relation replaces the
// causal order in A and P (page "Support TreeUpdateSolve kernel",
// trymirai/uzu PR #576).  No state carry is prepared.
// TCREC: the record's Wk, Qt, Kh and P as the tensor-core scan reads them
// (scan_tc.cu): each f32 region of n values holds n bf16 "hi" values, then n
// bf16 "lo" values (x - hi, rounded), in the K-major core-matrix order of a
// [rows][k] tile (8 rows x 8 k per 128-byte core matrix); same offsets and
// size as the f32 record.
template <typename Tin, bool TREE, bool TCREC>
__global__ void __launch_bounds__(kPrepThreads)
    gdr_chunk_prep(const Tin *__restrict__ q, const Tin *__restrict__ k,
                   const Tin *__restrict__ v, const float *__restrict__ g,
                   const float *__restrict__ beta, float *__restrict__ ws,
                   const int2 *__restrict__ chunks, const int *__restrict__ parents, int T,
                   int HK, int HV, int dk, int dv, int C, int NC, int g_scalar) {
    extern __shared__ float smem[];
    // padded rows: a warp's fragment loads hit distinct banks
    const int ldk = dk + 4, lda = C + 4, ldw = dk + dv + 8;
    float *Ks = smem;               // [C][ldk]
    float *Qs = Ks + C * ldk;       // [C][ldk]
    float *Gs = Qs + C * ldk;       // [C][ldk]
    float *As = Gs + C * ldk;       // [C][lda]
    float *Ws = As + C * lda;       // [C][ldw]: dk + dv columns used
    float *bs = Ws + C * ldw;       // [C]
    float *gmv = bs + C;            // [dk] G at the reference row
    float *egm = gmv + dk;          // [dk] exp(G_m)
    float *clv = egm + dk;          // [dk] exp(G_L - G_m)
    float *glv = clv + dk;          // [dk] G_L
    int *par = reinterpret_cast<int *>(glv + dk);                        // [C] (TREE)
    unsigned long long *anc = reinterpret_cast<unsigned long long *>(
        reinterpret_cast<uintptr_t>(par + C + 1) & ~(uintptr_t)7);     // [C] (TREE)

    // The chunk: its first token row in the [rows][H][d] view of the inputs,
    // its length, and its record.  Dense batches: CTA (b, hv, c), record
    // (b, hv, c).  Packed variable-length batches: CTA (chunk, hv) over the
    // table of every sequence's chunks {first row, length}, record (chunk, hv).
    int hv, L;
    size_t tr0, rec_idx;
    if (chunks) {
        const int ci = blockIdx.x / HV;
        hv = blockIdx.x % HV;
        const int2 e = chunks[ci];
        tr0 = (size_t)e.x;
        L = e.y;
        rec_idx = (size_t)ci * HV + hv;
    } else {
        const int c = blockIdx.x % NC;
        const int head_idx = blockIdx.x / NC;
        hv = head_idx % HV;
        const int b = head_idx / HV;
        tr0 = (size_t)b * T + (size_t)c * C;
        L = min(C, T - c * C);
        rec_idx = (size_t)head_idx * NC + c;
    }
    const int hk = hv / (HV / HK);
    const int tid = threadIdx.x;
    const ChunkLayout lay{C, dk, dv};
    float *rec = ws + rec_idx * lay.floats();

    // Load the chunk, four elements per access, several accesses in flight
    // per thread (rows >= L are zero; a zero gate keeps G flat there).
    {
        const int dk4 = dk / 4;
#pragma unroll 4
        for (int idx = tid; idx < C * dk4; idx += kPrepThreads) {
            const int r = idx / dk4, i = 4 * (idx % dk4);
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), qv = kv, gv = kv;
            if (r < L) {
                const size_t tk = (tr0 + r) * HK + hk;
                kv = load4(k + tk * dk + i);
                qv = load4(q + tk * dk + i);
                // a scalar gate has one log-decay per token and head
                if (g_scalar) {
                    const float x = g[(tr0 + r) * HV + hv];
                    gv = make_float4(x, x, x, x);
                } else {
                    gv = load4(g + ((tr0 + r) * HV + hv) * dk + i);
                }
            }
            *reinterpret_cast<float4 *>(Ks + r * ldk + i) = kv;
            *reinterpret_cast<float4 *>(Qs + r * ldk + i) = qv;
            *reinterpret_cast<float4 *>(Gs + r * ldk + i) = gv;
        }
    }
    for (int r = tid; r < C; r += kPrepThreads)
        bs[r] = r < L ? beta[(tr0 + r) * HV + hv] : 0.f;
    if (TREE) {
        const int b = blockIdx.x / NC / HV;
        for (int r = tid; r < C; r += kPrepThreads) par[r] = r < L ? parents[(size_t)b * T + r] : -1;
    }
    __syncthreads();

    if (TREE) {
        // Ancestor sets as bit masks (parents precede their children), and
        // the prefix sums of the log-decay along each token's root path.
        if (tid == 0) {
            for (int r = 0; r < C; ++r) {
                const int p = par[r];
                anc[r] = p < 0 ? 0ull : (anc[p] | (1ull << p));
            }
        }
        for (int i = tid; i < dk; i += kPrepThreads) {
            for (int r = 0; r < C; ++r) {
                const int p = par[r];
                Gs[r * ldk + i] += p < 0 ? 0.f : Gs[p * ldk + i];
            }
        }
    } else {
        // Per-channel inclusive prefix sum of the log-decay.
        for (int i = tid; i < dk; i += kPrepThreads) {
            float run = 0.f;
            for (int r = 0; r < C; ++r) {
                run += Gs[r * ldk + i];
                Gs[r * ldk + i] = run;
            }
        }
    }
    __syncthreads();

    // Reference-row factorisation (as in the tensor-core kernel): with m the
    // middle row of the chunk (a tree: its start, G_m = 0),
    //   A = tril(diag(beta) Lk R^T),  P = tril(Lq R^T),
    //   Lk = K e^{G - G_m}, Lq = Q e^{G - G_m}, R = K e^{G_m - G},
    // the decay leaves the dot products and A and P become 3xTF32 warp
    // products.  Taken when every factor stays within e^{80} (the spans
    // around m decay by at most 80 nats in every channel); otherwise A and P
    // come from the exact pairwise decays below.
    const int m = TREE ? -1 : (L - 1) / 2;
    bool in_range = true;
    if (tid < dk) {
        const int i = tid;
        const float gm = m < 0 ? 0.f : Gs[m * ldk + i];
        const float gl = Gs[(L - 1) * ldk + i];
        gmv[i] = gm;
        glv[i] = gl;
        egm[i] = expf(gm);
        clv[i] = expf(gl - gm);
        if (TREE) {
            float gmin = 0.f;
            for (int r = 0; r < L; ++r) gmin = fminf(gmin, Gs[r * ldk + i]);
            in_range = -gmin <= 80.f;
        } else {
            in_range = Gs[i] - gm <= 80.f && gm - gl <= 80.f;
        }
    }
    const bool fast = __syncthreads_and(in_range) != 0;
    float *Pg = rec + lay.p();
    const int lane = tid & 31, warp = tid >> 5;
    const int g8 = lane >> 2, t4 = lane & 3;
    if (fast) {
        // in place: Gs <- Lk, Qs <- Lq, Ks <- R
        for (int idx = tid; idx < C * dk; idx += kPrepThreads) {
            const int r = idx / dk, i = idx % dk;
            const float d = Gs[r * ldk + i] - gmv[i];
            const float up = expf(d), down = expf(-d);
            const float kv = Ks[r * ldk + i];
            Gs[r * ldk + i] = kv * up;
            Qs[r * ldk + i] *= up;
            Ks[r * ldk + i] = kv * down;
        }
        __syncthreads();
        // warp w: row tile w / 2 of A (w even) or P (w odd), every column
        // tile up to the diagonal block
        const int mt = warp >> 1;
        if (16 * mt < C) {
            const bool is_p = warp & 1;
            const float *Lx = is_p ? Qs : Gs;
            const int m0 = 16 * mt, ntn = 2 * mt + 2;
            float acc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
            for (int k0 = 0; k0 < dk; k0 += 8) {
                uint32_t ah[4], al[4];
                load_a3<false>(ah, al, Lx, ldk, m0, k0, 1.f, g8, t4);
#pragma unroll
                for (int n = 0; n < 8; ++n)
                    if (n < ntn) mma3_b<true>(acc[n], ah, al, Ks, ldk, k0, 8 * n, g8, t4);
            }
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                if (n >= ntn) continue;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = m0 + g8 + 8 * (e >> 1), sc = 8 * n + 2 * t4 + (e & 1);
                    const bool below = TREE ? (sc < r && ((anc[r] >> sc) & 1ull)) : sc < r;
                    if (is_p)
                        Pg[r * C + sc] = ((below || sc == r) && r < L) ? acc[n][e] : 0.f;
                    else
                        As[r * lda + sc] = (below && r < L) ? bs[r] * acc[n][e] : 0.f;
                }
            }
        }
    } else {
        // exact pairwise decays, every exponent <= 0
        for (int idx = tid; idx < C * C; idx += kPrepThreads) {
            const int r = idx / C, s = idx % C;
            // s is an earlier token r depends on: s <= r, or in a tree s == r
            // or an ancestor of r
            const bool below = TREE ? (s < r && ((anc[r] >> s) & 1ull)) : s < r;
            float a = 0.f, pp = 0.f;
            if ((below || s == r) && r < L) {
                const float *kr = Ks + r * ldk, *ks = Ks + s * ldk, *qr = Qs + r * ldk;
                const float *gr = Gs + r * ldk, *gs = Gs + s * ldk;
                for (int i = 0; i < dk; ++i) {
                    const float e = expf(gr[i] - gs[i]);
                    const float kse = ks[i] * e;
                    a = fmaf(kr[i], kse, a);
                    pp = fmaf(qr[i], kse, pp);
                }
            }
            As[r * lda + s] = below ? bs[r] * a : 0.f;
            Pg[idx] = pp;
        }
    }
    // Right-hand sides of the WY solve: diag(beta) [exp(G) * K | V]
    // (exp(G) K = Lk exp(G_m) on the factored path).
    const int nw = dk + dv;
    for (int idx = tid; idx < C * dk; idx += kPrepThreads) {
        const int r = idx / dk, col = idx % dk;
        float x = 0.f;
        if (r < L)
            x = fast ? bs[r] * Gs[r * ldk + col] * egm[col]
                     : bs[r] * Ks[r * ldk + col] * expf(Gs[r * ldk + col]);
        Ws[r * ldw + col] = x;
    }
    {
        const int dv4 = dv / 4;
#pragma unroll 4
        for (int idx = tid; idx < C * dv4; idx += kPrepThreads) {
            const int r = idx / dv4, j = 4 * (idx % dv4);
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < L) {
                x = load4(v + ((tr0 + r) * HV + hv) * dv + j);
                const float br = bs[r];
                x.x *= br; x.y *= br; x.z *= br; x.w *= br;
            }
            *reinterpret_cast<float4 *>(Ws + r * ldw + dk + j) = x;
        }
    }
    __syncthreads();

    // (I + A) W = RHS, block by block of 16 rows: first the rows' update by
    // the blocks already solved, W_I -= A_IJ W_J (J < I), as 3xTF32 warp
    // products (warp w: column tiles 4w .. 4w + 3 of the dk + dv columns),
    // then the unit-lower 16 x 16 diagonal block by forward substitution, one
    // column per thread.  Rows past L have zero right-hand sides and zero
    // rows of A, so their W stays zero.
    for (int I = 0; 16 * I < L; ++I) {
        const int r0 = 16 * I;
        if (I > 0) {
            // warp w: column tiles 4w .. 4w + 3 (all four exist whenever the
            // first does: dk + dv is a multiple of 32)
            const int nbase = 32 * warp;
            if (nbase < nw) {
                float acc[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int n0 = nbase + 8 * nt;
                    acc[nt][0] = Ws[(r0 + g8) * ldw + n0 + 2 * t4];
                    acc[nt][1] = Ws[(r0 + g8) * ldw + n0 + 2 * t4 + 1];
                    acc[nt][2] = Ws[(r0 + g8 + 8) * ldw + n0 + 2 * t4];
                    acc[nt][3] = Ws[(r0 + g8 + 8) * ldw + n0 + 2 * t4 + 1];
                }
                mma3_rows<4, false>(acc, As, lda, r0, r0, Ws, ldw, nbase, -1.f, g8, t4);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const int n0 = nbase + 8 * nt;
                    Ws[(r0 + g8) * ldw + n0 + 2 * t4] = acc[nt][0];
                    Ws[(r0 + g8) * ldw + n0 + 2 * t4 + 1] = acc[nt][1];
                    Ws[(r0 + g8 + 8) * ldw + n0 + 2 * t4] = acc[nt][2];
                    Ws[(r0 + g8 + 8) * ldw + n0 + 2 * t4 + 1] = acc[nt][3];
                }
            }
            __syncthreads();
        }
        for (int col = tid; col < nw; col += kPrepThreads) {
            float w[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) w[r] = Ws[(r0 + r) * ldw + col];
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                const float *ar = As + (r0 + r) * lda + r0;
#pragma unroll
                for (int q = 0; q < r; ++q) w[r] = fmaf(-ar[q], w[q], w[r]);
            }
#pragma unroll
            for (int r = 1; r < 16; ++r) Ws[(r0 + r) * ldw + col] = w[r];
        }
        __syncthreads();
    }

    // Scan operands: Wk, Wv, Qt = exp(G) Q, Kh = exp(G_L - G) K, gam = exp(G_L)
    // (a tree has no last token to carry the state to: no Kh, gam).  On the
    // factored path Qs holds Lq and Ks holds R: Qt = Lq exp(G_m) and
    // Kh = R exp(G_L - G_m).
    // a value into a TC-layout region of a [rows][kext] tile: hi, then lo
    auto put_tc = [&](size_t region, int row, int kk, int kext, int rows, float x) {
        __nv_bfloat16 *base = reinterpret_cast<__nv_bfloat16 *>(rec + region);
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        const uint32_t o = sm100::kmajor_off(row, kk, kext) / 2;
        base[o] = h;
        base[(size_t)rows * kext + o] = __float2bfloat16_rn(x - __bfloat162float(h));
    };
    for (int idx = tid; idx < C * dk; idx += kPrepThreads) {
        const int r = idx / dk, i = idx % dk;
        float qt, kh = 0.f;
        if (fast) {
            qt = Qs[r * ldk + i] * egm[i];
            if (!TREE) kh = r < L ? Ks[r * ldk + i] * clv[i] : 0.f;
        } else {
            const float gri = Gs[r * ldk + i];
            qt = Qs[r * ldk + i] * expf(gri);
            if (!TREE) kh = r < L ? Ks[r * ldk + i] * expf(glv[i] - gri) : 0.f;
        }
        if (TCREC) {
            put_tc(lay.wk(), r, i, dk, C, Ws[r * ldw + i]);
            put_tc(lay.qt(), r, i, dk, C, qt);
            put_tc(lay.kh(), r, i, dk, C, kh);
        } else {
            rec[lay.wk() + idx] = Ws[r * ldw + i];
            rec[lay.qt() + idx] = qt;
            if (!TREE) rec[lay.kh() + idx] = kh;
        }
    }
    if (TCREC) {
        // P, written above as f32 rows up to each row tile's diagonal block,
        // into the same region in TC layout with zeros above the diagonal
        // (the tensor-core products run over every column): every thread
        // holds its values before any is overwritten
        constexpr int kMaxPer = 64 * 64 / kPrepThreads;
        float pv[kMaxPer];
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kMaxPer; ++m) {
            const int idx = tid + kPrepThreads * m;
            pv[m] = (idx < C * C && idx % C <= idx / C) ? Pg[idx] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kMaxPer; ++m) {
            const int idx = tid + kPrepThreads * m;
            if (idx < C * C) put_tc(lay.p(), idx / C, idx % C, C, C, pv[m]);
        }
    }
    for (int idx = tid; idx < C * dv / 4; idx += kPrepThreads) {
        const int r = (4 * idx) / dv, j = (4 * idx) % dv;
        *reinterpret_cast<float4 *>(rec + lay.wv() + r * dv + j) =
            *reinterpret_cast<const float4 *>(Ws + r * ldw + dk + j);
    }
    if (!TREE)
        for (int i = tid; i < dk; i += kPrepThreads) rec[lay.gam() + i] = expf(glv[i]);
}

// TREE: one chunk (the tree), outputs only: no state update, no ht.
//
// Shared-memory rows are padded so that the fragment loads of a warp fall in
// distinct banks: A operands by 4 floats (dk + 4, C + 4), B operands to 40
// (32 columns + 8).  Per chunk, with 8 warps: U = Wv - Wk S (4 x 4 tiles,
// warp w: row tile w / 2, column tiles 2 (w % 2) and +1), O = Qt S + P U
// (same tiles), then S = diag(gam) S + Kh^T U (8 x 4 tiles, warp w: row
// tile w, all four column tiles).
template <typename Tin, bool TREE>
__global__ void __launch_bounds__(kScanThreads)
    gdr_chunk_scan(const float *__restrict__ ws, const float *h0, Tin *__restrict__ out,
                   float *ht, const int4 *__restrict__ seqs, int T_dense, int HV, int dk, int dv,
                   int C, int NC_dense) {
    extern __shared__ float smem[];
    constexpr int ldb = kScanBV + 8;     // B-operand rows (S, U)
    const int lda = dk + 4;              // A-operand rows over dk (Wk, Qt, Kh)
    const int ldp = C + 4;               // P rows
    float *Ss = smem;                    // [dk][ldb]  state tile
    float *Wk = Ss + dk * ldb;           // [C][lda]
    float *Qt = Wk + C * lda;            // [C][lda]
    float *Kh = Qt + C * lda;            // [C][lda]
    float *Ps = Kh + C * lda;            // [C][ldp]
    float *Us = Ps + C * ldp;            // [C][ldb]
    float *Wv = Us + C * ldb;            // [C][BV]
    float *gam = Wv + C * kScanBV;       // [dk]

    const int ntile = dv / kScanBV;
    const int tile = blockIdx.x % ntile;
    const int hv = (blockIdx.x / ntile) % HV;
    const int b = blockIdx.x / ntile / HV;
    // The sequence: first token row, length, state slot, and where its chunk
    // records start and how far apart they are (dense: b's own rows, slot b,
    // records (b, hv, c); packed: {first row, length, slot, first chunk}
    // from the table, records (chunk, hv)).
    size_t tok0 = (size_t)b * T_dense, rec0 = ((size_t)b * HV + hv) * NC_dense, rec_step = 1;
    int T = T_dense, slot = b;
    if (seqs) {
        const int4 sd = seqs[b];
        tok0 = (size_t)sd.x;
        T = sd.y;
        slot = sd.z;
        rec0 = (size_t)sd.w * HV + hv;
        rec_step = HV;
    }
    const int NC = (T + C - 1) / C;
    const size_t head_idx = (size_t)slot * HV + hv;  // state slot
    const int j0 = tile * kScanBV;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const ChunkLayout lay{C, dk, dv};

    for (int idx = tid; idx < dk * kScanBV; idx += kScanThreads) {
        const int i = idx / kScanBV, j = idx % kScanBV;
        Ss[i * ldb + j] = h0 ? h0[(head_idx * dk + i) * dv + j0 + j] : 0.f;
    }

    for (int c = 0; c < NC; ++c) {
        const float *rec = ws + (rec0 + (size_t)c * rec_step) * lay.floats();
        const int t0 = c * C;
        const int L = min(C, T - t0);
        // the chunk's record, 16-byte asynchronous copies all in flight at
        // once (every part starts on a multiple of 4 floats)
        const int dk4 = dk / 4;
        for (int idx = tid; idx < C * dk4; idx += kScanThreads) {
            const int r = idx / dk4, i = 4 * (idx % dk4);
            cp_async16(Wk + r * lda + i, rec + lay.wk() + r * dk + i);
            cp_async16(Qt + r * lda + i, rec + lay.qt() + r * dk + i);
            if (!TREE) cp_async16(Kh + r * lda + i, rec + lay.kh() + r * dk + i);
        }
        for (int idx = tid; idx < C * C / 4; idx += kScanThreads) {
            const int r = (4 * idx) / C, s4 = (4 * idx) % C;
            cp_async16(Ps + r * ldp + s4, rec + lay.p() + r * C + s4);
        }
        for (int idx = tid; idx < C * kScanBV / 4; idx += kScanThreads) {
            const int r = (4 * idx) / kScanBV, j = (4 * idx) % kScanBV;
            cp_async16(Wv + r * kScanBV + j, rec + lay.wv() + (size_t)r * dv + j0 + j);
        }
        if (!TREE)
            for (int i = 4 * tid; i < dk; i += 4 * kScanThreads) cp_async16(gam + i, rec + lay.gam() + i);
        cp_async_wait_all_copies();
        __syncthreads();

        // U = Wv - Wk S0 (rows past L are zero: Wk and Wv are)
        const int um0 = 16 * (warp >> 1), unb = 16 * (warp & 1);
        if (um0 < C) {
            float acc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int n0 = unb + 8 * nt;
                acc[nt][0] = Wv[(um0 + g) * kScanBV + n0 + 2 * t];
                acc[nt][1] = Wv[(um0 + g) * kScanBV + n0 + 2 * t + 1];
                acc[nt][2] = Wv[(um0 + g + 8) * kScanBV + n0 + 2 * t];
                acc[nt][3] = Wv[(um0 + g + 8) * kScanBV + n0 + 2 * t + 1];
            }
            mma3_rows<2, false>(acc, Wk, lda, um0, dk, Ss, ldb, unb, -1.f, g, t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int n0 = unb + 8 * nt;
                Us[(um0 + g) * ldb + n0 + 2 * t] = acc[nt][0];
                Us[(um0 + g) * ldb + n0 + 2 * t + 1] = acc[nt][1];
                Us[(um0 + g + 8) * ldb + n0 + 2 * t] = acc[nt][2];
                Us[(um0 + g + 8) * ldb + n0 + 2 * t + 1] = acc[nt][3];
            }
        }
        __syncthreads();

        // O = Qt S0 + P U (P is zero above the diagonal and off a tree's
        // ancestors), rows below L stored
        if (um0 < C) {
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            mma3_rows<2, false>(acc, Qt, lda, um0, dk, Ss, ldb, unb, 1.f, g, t);
            mma3_rows<2, false>(acc, Ps, ldp, um0, um0 + 16, Us, ldb, unb, 1.f, g, t);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int n0 = unb + 8 * nt;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = um0 + g + 8 * h;
                    if (r < L) {
                        Tin *o = out + ((tok0 + t0 + r) * HV + hv) * dv + j0 + n0 + 2 * t;
                        o[0] = from_f32<Tin>(acc[nt][2 * h]);
                        o[1] = from_f32<Tin>(acc[nt][2 * h + 1]);
                    }
                }
            }
        }

        if (TREE) break;  // one chunk; no state to carry
        // S = diag(gam) S0 + Kh^T U (rows of Kh and U past L are zero), kept
        // in registers until every warp is done reading S0
        float sacc[4][4];
        const int sm0 = 16 * warp;
        const bool s_rows = sm0 < dk;
        if (s_rows) {
            const float ga = gam[sm0 + g], gb = gam[sm0 + g + 8];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int n0 = 8 * nt;
                sacc[nt][0] = ga * Ss[(sm0 + g) * ldb + n0 + 2 * t];
                sacc[nt][1] = ga * Ss[(sm0 + g) * ldb + n0 + 2 * t + 1];
                sacc[nt][2] = gb * Ss[(sm0 + g + 8) * ldb + n0 + 2 * t];
                sacc[nt][3] = gb * Ss[(sm0 + g + 8) * ldb + n0 + 2 * t + 1];
            }
            mma3_rows<4, true>(sacc, Kh, lda, sm0, L, Us, ldb, 0, 1.f, g, t);
        }
        __syncthreads();
        if (s_rows) {
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int n0 = 8 * nt;
                Ss[(sm0 + g) * ldb + n0 + 2 * t] = sacc[nt][0];
                Ss[(sm0 + g) * ldb + n0 + 2 * t + 1] = sacc[nt][1];
                Ss[(sm0 + g + 8) * ldb + n0 + 2 * t] = sacc[nt][2];
                Ss[(sm0 + g + 8) * ldb + n0 + 2 * t + 1] = sacc[nt][3];
            }
        }
        __syncthreads();
    }

    if (!TREE && ht) {
        for (int idx = tid; idx < dk * kScanBV; idx += kScanThreads) {
            const int i = idx / kScanBV, j = idx % kScanBV;
            ht[(head_idx * dk + i) * dv + j0 + j] = Ss[i * ldb + j];
        }
    }
}

size_t prep_smem_bytes(int dk, int dv, int C) {
    // floats, then (trees) C parent indices and C 8-byte ancestor masks
    return sizeof(float) * ((size_t)3 * C * (dk + 4) + (size_t)C * (C + 4) +
                            (size_t)C * (dk + dv + 8) + C + (size_t)4 * dk) +
           sizeof(int) * (C + 2) + sizeof(unsigned long long) * C;
}
size_t scan_smem_bytes(int dk, int C) {
    const size_t ldb = kScanBV + 8;
    return sizeof(float) * ((size_t)dk * ldb + (size_t)3 * C * (dk + 4) + (size_t)C * (C + 4) +
                            (size_t)C * ldb + (size_t)C * kScanBV + dk);
}

// Dense batches: chunks == seqs == nullptr, B x T from p.  Packed batches:
// nchunks chunk records and p.B sequence records.  Trees (TREE): p.T <=
// p.chunk tokens per batch element, parents [B][T] on the device.
// TCREC: a segmented scan (SegScan::P >= 2) runs `n` more sequences after
// the p.B whole ones (none for a dense batch cut into segments).
struct SegScan {
    const ScanSeq *seqs = nullptr;
    int n = 0, P = 0;
    void *ws = nullptr;
    bool whole = true;  // the p.B sequences of the batch walk whole
};

template <typename Tin, bool TREE, bool TCREC = false>
cudaError_t launch_generic_t(const Problem &p, void *workspace, const int2 *chunks, int nchunks,
                             const int4 *seqs, const int *parents, cudaStream_t stream,
                             const SegScan &seg = SegScan{}) {
    const int C = p.chunk;
    const int NC = (p.T + C - 1) / C;
    float *ws = static_cast<float *>(workspace);
    const long long prep_blocks = chunks ? (long long)nchunks * p.HV : (long long)p.B * p.HV * NC;
    const long long scan_blocks = (long long)p.B * p.HV * (p.dv / kScanBV);
    if (prep_blocks > 0x7fffffffLL || scan_blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t sp = prep_smem_bytes(p.dk, p.dv, C);
    const size_t ss = scan_smem_bytes(p.dk, C);
    cudaError_t e;
    if (TCREC && !TREE && prep_tc_supported(p)) {
        // the prep on the tensor cores, then the scan below
        const ChunkLayout lay{C, p.dk, p.dv};
        e = launch_chunk_prep_tc(p, ws, lay.floats(), chunks, nchunks, stream);
        if (e != cudaSuccess) return e;
        if (seg.whole) {
            e = launch_chunk_scan_tc(p, ws, lay.floats(), seqs, p.B, stream);
            if (e != cudaSuccess) return e;
        }
        if (seg.P >= 2 && seg.n > 0)
            e = launch_scan_segmented(p, ws, lay.floats(), seg.seqs, seg.n, seg.P, seg.ws, stream);
        return e;
    }
    e = cudaFuncSetAttribute(gdr_chunk_prep<Tin, TREE, TCREC>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gdr_chunk_scan<Tin, TREE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ss);
    if (e != cudaSuccess) return e;
    trace_begin(kKernChunkPrep, stream);
    gdr_chunk_prep<Tin, TREE, TCREC><<<(unsigned)prep_blocks, kPrepThreads, sp, stream>>>(
        static_cast<const Tin *>(p.q), static_cast<const Tin *>(p.k),
        static_cast<const Tin *>(p.v), p.g, p.beta, ws, chunks, parents, p.T, p.HK, p.HV, p.dk,
        p.dv, C, NC, p.g_scalar);
    trace_end(kKernChunkPrep, stream);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (TCREC) {
        const ChunkLayout lay{C, p.dk, p.dv};
        if (seg.whole) {
            e = launch_chunk_scan_tc(p, ws, lay.floats(), seqs, p.B, stream);
            if (e != cudaSuccess) return e;
        }
        if (seg.P >= 2 && seg.n > 0)
            e = launch_scan_segmented(p, ws, lay.floats(), seg.seqs, seg.n, seg.P, seg.ws, stream);
        return e;
    }
    trace_begin(kKernChunkScan, stream);
    gdr_chunk_scan<Tin, TREE><<<(unsigned)scan_blocks, kScanThreads, ss, stream>>>(
        ws, p.h0, static_cast<Tin *>(p.out), p.ht, seqs, p.T, p.HV, p.dk, p.dv, C, NC);
    trace_end(kKernChunkScan, stream);
    return cudaGetLastError();
}

}  // namespace

size_t generic_prefill_workspace_bytes(const Problem &p) {
    const int NC = (p.T + p.chunk - 1) / p.chunk;
    const ChunkLayout lay{p.chunk, p.dk, p.dv};
    return sizeof(float) * lay.floats() * (size_t)p.B * p.HV * NC;
}

size_t generic_prefill_workspace_bytes(const Problem &p, int segments) {
    const size_t rec = generic_prefill_workspace_bytes(p);
    if (segments < 2) return rec;
    return ((rec + 255) & ~(size_t)255) + scan_segmented_bytes(p, p.B, segments);
}

cudaError_t launch_generic_prefill(const Problem &p, void *workspace, cudaStream_t stream,
                                   bool tc_scan, int segments) {
    if (tc_scan && segments >= 2) {
        // every batch element cut into segments after the prep
        const int NC = (p.T + p.chunk - 1) / p.chunk;
        std::vector<ScanSeq> list((size_t)p.B);
        for (int b = 0; b < p.B; ++b)
            list[b] = ScanSeq{(long long)b * p.T, (long long)b * p.HV * NC, p.T, b, NC, 1};
        SegScan seg;
        seg.seqs = list.data();
        seg.n = p.B;
        seg.P = segments;
        seg.ws = static_cast<unsigned char *>(workspace) +
                 ((generic_prefill_workspace_bytes(p) + 255) & ~(size_t)255);
        seg.whole = false;
        return p.bf16 ? launch_generic_t<__nv_bfloat16, false, true>(p, workspace, nullptr, 0,
                                                                     nullptr, nullptr, stream, seg)
                      : launch_generic_t<float, false, true>(p, workspace, nullptr, 0, nullptr,
                                                             nullptr, stream, seg);
    }
    if (tc_scan)
        return p.bf16 ? launch_generic_t<__nv_bfloat16, false, true>(p, workspace, nullptr, 0,
                                                                     nullptr, nullptr, stream)
                      : launch_generic_t<float, false, true>(p, workspace, nullptr, 0, nullptr,
                                                             nullptr, stream);
    return p.bf16 ? launch_generic_t<__nv_bfloat16, false>(p, workspace, nullptr, 0, nullptr,
                                                           nullptr, stream)
                  : launch_generic_t<float, false>(p, workspace, nullptr, 0, nullptr, nullptr,
                                                   stream);
}

size_t generic_varlen_record_bytes(const Problem &p, long long nchunks) {
    const ChunkLayout lay{p.chunk, p.dk, p.dv};
    return sizeof(float) * lay.floats() * (size_t)nchunks * p.HV;
}

cudaError_t launch_generic_prefill_varlen(const Problem &p, void *records, const int2 *chunks,
                                          int nchunks, const int4 *seqs, cudaStream_t stream,
                                          bool tc_scan, const ScanSeq *seg_seqs, int nseg,
                                          int seg_P, void *seg_ws) {
    if (tc_scan) {
        SegScan seg;
        seg.seqs = seg_seqs;
        seg.n = nseg;
        seg.P = seg_P;
        seg.ws = seg_ws;
        seg.whole = p.B > 0;
        return p.bf16 ? launch_generic_t<__nv_bfloat16, false, true>(p, records, chunks, nchunks,
                                                                     seqs, nullptr, stream, seg)
                      : launch_generic_t<float, false, true>(p, records, chunks, nchunks, seqs,
                                                             nullptr, stream, seg);
    }
    return p.bf16 ? launch_generic_t<__nv_bfloat16, false>(p, records, chunks, nchunks, seqs,
                                                           nullptr, stream)
                  : launch_generic_t<float, false>(p, records, chunks, nchunks, seqs, nullptr,
                                                   stream);
}

size_t generic_tree_record_bytes(const Problem &p) {
    const ChunkLayout lay{p.chunk, p.dk, p.dv};
    return sizeof(float) * lay.floats() * (size_t)p.B * p.HV;
}

cudaError_t launch_generic_tree(const Problem &p, void *records, const int *parents,
                                cudaStream_t stream) {
    return p.bf16 ? launch_generic_t<__nv_bfloat16, true>(p, records, nullptr, 0, nullptr,
                                                          parents, stream)
                  : launch_generic_t<float, true>(p, records, nullptr, 0, nullptr, parents,
                                                  stream);
}

}  // namespace gdr
