// k_hash.cu -- on-device per-step state hash.
//
// The pages record a hash of the training state after every optimiser step so
// that a replay can be checked against the run; they hash on the host (about
// 6 s per step) and name on-device hashing as future work (Open-1B review,
// onedev.kr/papers/92, section "Premises and limits"; rit.work blog
// "open-1b-auditable-training", paragraph 4).  The construction here is the
// Merkle Tree Hash of RFC 6962 (section 2.1) over SHA-256 (FIPS 180-4):
//   leaves   = every buffer cut into REPRO_HASH_LEAF_BYTES pieces, buffer order;
//   leaf     = SHA-256(0x00 || leaf bytes);
//   node     = SHA-256(0x01 || left || right);
//   the tree pairs adjacent nodes level by level and carries an odd last node
//   up unchanged, which is RFC 6962's split at the largest power of two;
//   no leaves: SHA-256 of the empty string.
//
// SHA-256 is sequential within a message, so the parallelism is one leaf per
// thread (k_hash_leaves), then one node per thread per tree level
// (k_hash_level).  The compression function is ALU work (32-bit rotates,
// three-input logic, adds): the kernels are bound by the integer pipe, not
// by HBM.  Digests are stored as bytes in the standard (big-endian) order, so
// a node's input is the 64 contiguous bytes of its two children.
#include "internal.h"

namespace repro {
namespace {

__constant__ uint32_t kRound[64] = {
    0x428a2f98u, 0x71374491u, 0xb5c0fbcfu, 0xe9b5dba5u, 0x3956c25bu, 0x59f111f1u, 0x923f82a4u,
    0xab1c5ed5u, 0xd807aa98u, 0x12835b01u, 0x243185beu, 0x550c7dc3u, 0x72be5d74u, 0x80deb1feu,
    0x9bdc06a7u, 0xc19bf174u, 0xe49b69c1u, 0xefbe4786u, 0x0fc19dc6u, 0x240ca1ccu, 0x2de92c6fu,
    0x4a7484aau, 0x5cb0a9dcu, 0x76f988dau, 0x983e5152u, 0xa831c66du, 0xb00327c8u, 0xbf597fc7u,
    0xc6e00bf3u, 0xd5a79147u, 0x06ca6351u, 0x14292967u, 0x27b70a85u, 0x2e1b2138u, 0x4d2c6dfcu,
    0x53380d13u, 0x650a7354u, 0x766a0abbu, 0x81c2c92eu, 0x92722c85u, 0xa2bfe8a1u, 0xa81a664bu,
    0xc24b8b70u, 0xc76c51a3u, 0xd192e819u, 0xd6990624u, 0xf40e3585u, 0x106aa070u, 0x19a4c116u,
    0x1e376c08u, 0x2748774cu, 0x34b0bcb5u, 0x391c0cb3u, 0x4ed8aa4au, 0x5b9cca4fu, 0x682e6ff3u,
    0x748f82eeu, 0x78a5636fu, 0x84c87814u, 0x8cc70208u, 0x90befffau, 0xa4506cebu, 0xbef9a3f7u,
    0xc67178f2u};

__device__ __forceinline__ void init_state(uint32_t (&H)[8])
{
    H[0] = 0x6a09e667u;
    H[1] = 0xbb67ae85u;
    H[2] = 0x3c6ef372u;
    H[3] = 0xa54ff53au;
    H[4] = 0x510e527fu;
    H[5] = 0x9b05688cu;
    H[6] = 0x1f83d9abu;
    H[7] = 0x5be0cd19u;
}

__device__ __forceinline__ uint32_t rotr(uint32_t x, int n)
{
    return __funnelshift_r(x, x, n);
}

// one compression of a 16-word (big-endian words) message block
__device__ __forceinline__ void compress(uint32_t (&H)[8], uint32_t (&W)[16])
{
    uint32_t a = H[0], b = H[1], c = H[2], d = H[3], e = H[4], f = H[5], g = H[6], h = H[7];
#pragma unroll
    for (int t = 0; t < 64; ++t) {
        uint32_t w;
        if (t < 16) {
            w = W[t];
        } else {
            const uint32_t x15 = W[(t - 15) & 15], x2 = W[(t - 2) & 15];
            const uint32_t s0 = rotr(x15, 7) ^ rotr(x15, 18) ^ (x15 >> 3);
            const uint32_t s1 = rotr(x2, 17) ^ rotr(x2, 19) ^ (x2 >> 10);
            w = W[t & 15] = W[t & 15] + s0 + W[(t - 7) & 15] + s1;
        }
        const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
        const uint32_t ch = (e & f) ^ (~e & g);
        const uint32_t t1 = h + S1 + ch + kRound[t] + w;
        const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
        const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
        const uint32_t t2 = S0 + maj;
        h = g;
        g = f;
        f = e;
        e = d + t1;
        d = c;
        c = b;
        b = a;
        a = t1 + t2;
    }
    H[0] += a;
    H[1] += b;
    H[2] += c;
    H[3] += d;
    H[4] += e;
    H[5] += f;
    H[6] += g;
    H[7] += h;
}

// SHA-256 of (prefix byte || data[0 .. L)); data 16-byte aligned
__device__ void sha256_prefixed(uint32_t prefix, const uint8_t* __restrict__ data, int64_t L,
                                uint32_t (&H)[8])
{
    init_state(H);
    // whole message blocks: message byte 64b + j is data[64b + j - 1] (the
    // prefix for j = 0 of block 0), so word w is the last byte of data word
    // w-1 followed by the first three bytes of data word w
    const int64_t nfull = L >> 6;
    uint32_t prev = prefix << 24;
    for (int64_t blk = 0; blk < nfull; ++blk) {
        const uint4* p = reinterpret_cast<const uint4*>(data + (blk << 6));
        uint32_t d[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint4 v = __ldg(p + u);
            d[4 * u] = v.x;
            d[4 * u + 1] = v.y;
            d[4 * u + 2] = v.z;
            d[4 * u + 3] = v.w;
        }
        uint32_t W[16];
        W[0] = __byte_perm(prev, d[0], 0x3456);
#pragma unroll
        for (int w = 1; w < 16; ++w)
            W[w] = __byte_perm(d[w - 1], d[w], 0x3456);
        prev = d[15];
        compress(H, W);
    }
    // the rest of the message, the 0x80 terminator, zeros and the 64-bit
    // big-endian bit length, in one or two blocks
    const int64_t total = L + 1;
    const int64_t base = nfull << 6;
    const int rem = (int)(total - base);            // 1 .. 64
    const int nblk = rem + 9 <= 64 ? 1 : 2;
    const uint64_t bits = (uint64_t)total * 8u;
    for (int bk = 0; bk < nblk; ++bk) {
        uint32_t W[16];
        for (int w = 0; w < 16; ++w) {
            uint32_t word = 0;
            for (int k = 0; k < 4; ++k) {
                const int64_t i = base + 64 * bk + 4 * w + k;
                uint32_t byte = 0;
                if (i < total)
                    byte = i == 0 ? prefix : (uint32_t)data[i - 1];
                else if (i == total)
                    byte = 0x80u;
                word = (word << 8) | byte;
            }
            W[w] = word;
        }
        if (bk == nblk - 1) {
            W[14] = (uint32_t)(bits >> 32);
            W[15] = (uint32_t)bits;
        }
        compress(H, W);
    }
}

// digest words as bytes in the standard order
__device__ __forceinline__ void store_digest(uint32_t* __restrict__ out, const uint32_t (&H)[8])
{
    uint4* o = reinterpret_cast<uint4*>(out);
    o[0] = make_uint4(__byte_perm(H[0], 0, 0x0123), __byte_perm(H[1], 0, 0x0123),
                      __byte_perm(H[2], 0, 0x0123), __byte_perm(H[3], 0, 0x0123));
    o[1] = make_uint4(__byte_perm(H[4], 0, 0x0123), __byte_perm(H[5], 0, 0x0123),
                      __byte_perm(H[6], 0, 0x0123), __byte_perm(H[7], 0, 0x0123));
}

struct HashBufs {
    const uint8_t* ptr[REPRO_MAX_PARTS_INTERNAL];
    int64_t nbytes[REPRO_MAX_PARTS_INTERNAL];
    int64_t first_leaf[REPRO_MAX_PARTS_INTERNAL + 1];
    int nbuf;
};

__global__ void __launch_bounds__(128)
    k_hash_leaves(const HashBufs bufs, int64_t nleaves, int64_t leaf_bytes, uint32_t* __restrict__ out)
{
    const int64_t leaf = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (leaf >= nleaves)
        return;
    int b = 0;   // the buffer holding this leaf (empty buffers are skipped)
    while (b + 1 < bufs.nbuf && bufs.first_leaf[b + 1] <= leaf)
        ++b;
    const int64_t off = (leaf - bufs.first_leaf[b]) * leaf_bytes;
    const int64_t rest = bufs.nbytes[b] - off;
    uint32_t H[8];
    sha256_prefixed(0x00u, bufs.ptr[b] + off, rest < leaf_bytes ? rest : leaf_bytes, H);
    store_digest(out + 8 * leaf, H);
}

// one tree level: node j = SHA-256(0x01 || in[2j] || in[2j+1]), or in[2j]
// carried when it has no right sibling
__global__ void __launch_bounds__(128)
    k_hash_level(const uint32_t* __restrict__ in, int64_t count, uint32_t* __restrict__ out)
{
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (2 * j >= count)
        return;
    if (2 * j + 1 < count) {
        uint32_t H[8];
        sha256_prefixed(0x01u, reinterpret_cast<const uint8_t*>(in + 16 * j), 64, H);
        store_digest(out + 8 * j, H);
    } else {
        const uint4* s = reinterpret_cast<const uint4*>(in + 16 * j);
        uint4* o = reinterpret_cast<uint4*>(out + 8 * j);
        o[0] = s[0];
        o[1] = s[1];
    }
}

// no leaves: SHA-256 of the empty message
__global__ void k_hash_empty(uint32_t* __restrict__ out)
{
    uint32_t H[8], W[16];
    init_state(H);
    for (int w = 0; w < 16; ++w)
        W[w] = 0;
    W[0] = 0x80000000u;
    compress(H, W);
    store_digest(out, H);
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t align256(int64_t b) { return (b + 255) & ~(int64_t)255; }

} // namespace

int64_t hash_leaf_count(const int64_t* nbytes, int nbuf, int64_t leaf_bytes)
{
    int64_t n = 0;
    for (int b = 0; b < nbuf; ++b)
        n += cdiv(nbytes[b], leaf_bytes);
    return n;
}

size_t hash_ws_bytes(int64_t nleaves)
{
    if (nleaves <= 1)
        return 0;
    return (size_t)(align256(nleaves * 32) + align256(cdiv(nleaves, 2) * 32));
}

cudaError_t launch_state_hash(const void* const* bufs, const int64_t* nbytes, int nbuf,
                              int64_t leaf_bytes, uint8_t* digest, void* ws, cudaStream_t st)
{
    uint32_t* dig = reinterpret_cast<uint32_t*>(digest);
    const int64_t nleaves = hash_leaf_count(nbytes, nbuf, leaf_bytes);
    if (nleaves == 0) {
        k_hash_empty<<<1, 1, 0, st>>>(dig);
        count_launches(1);
        return cudaGetLastError();
    }
    HashBufs hb;
    hb.nbuf = nbuf;
    hb.first_leaf[0] = 0;
    for (int b = 0; b < nbuf; ++b) {
        hb.ptr[b] = static_cast<const uint8_t*>(bufs[b]);
        hb.nbytes[b] = nbytes[b];
        hb.first_leaf[b + 1] = hb.first_leaf[b] + cdiv(nbytes[b], leaf_bytes);
    }
    uint32_t* A = static_cast<uint32_t*>(ws);
    uint32_t* B = nleaves > 1
                      ? reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + align256(nleaves * 32))
                      : nullptr;
    k_hash_leaves<<<(unsigned)cdiv(nleaves, 128), 128, 0, st>>>(hb, nleaves, leaf_bytes,
                                                                 nleaves == 1 ? dig : A);
    count_launches(1);
    int64_t count = nleaves;
    uint32_t* cur = A;
    uint32_t* nxt = B;
    while (count > 1) {
        const int64_t up = cdiv(count, 2);
        uint32_t* dst = up == 1 ? dig : nxt;
        k_hash_level<<<(unsigned)cdiv(up, 128), 128, 0, st>>>(cur, count, dst);
        count_launches(1);
        count = up;
        uint32_t* t = cur;
        cur = nxt;
        nxt = t;
    }
    return cudaGetLastError();
}

} // namespace repro
