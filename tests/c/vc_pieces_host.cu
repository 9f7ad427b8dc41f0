// Host-side check of the library's misaligned 16-byte accesses (the helpers
// in vc_device.cuh that reach shards off the 16-byte grid; they are
// __host__ __device__): for every element size and every offset a vector
// of that element size can sit at, st_aligned writes exactly its 16 bytes
// and leaves every other byte alone, ld_aligned returns exactly the 16
// bytes at its address, st_bytes writes exactly the byte range it is given,
// and ld_block_part returns exactly the part of the block it is given with
// zeros elsewhere (the partial blocks of the warp-realigned accesses).  The
// expected bytes are computed here one byte at a time.  Built with nvcc,
// run on the CPU; prints "ok" or the failures and exits non-zero.
#include <cstdio>
#include <cstring>

#include "vc_device.cuh"

namespace {

int failures = 0;

void fail(const char* what, int es, int d, int byte) {
    if (failures++ < 10) std::printf("FAIL %s es=%d d=%d byte=%d\n", what, es, d, byte);
}

unsigned lcg(unsigned& s) {
    s = s * 1664525u + 1013904223u;
    return s >> 8;
}

uint4 random_vec(unsigned& s) {
    return make_uint4(lcg(s) ^ (lcg(s) << 16), lcg(s) ^ (lcg(s) << 16), lcg(s) ^ (lcg(s) << 16),
                      lcg(s) ^ (lcg(s) << 16));
}

void vec_bytes(const uint4& v, unsigned char (&b)[16]) {
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
    for (int k = 0; k < 16; ++k) b[k] = (unsigned char)(w[k / 4] >> (8 * (k % 4)));
}

template <int ES>
void check_es(unsigned& seed) {
    alignas(16) unsigned char buf[64];
    unsigned char* blk = buf + 16;  // 16-byte aligned
    for (int d = 0; d < 16; d += ES) {
        for (int rep = 0; rep < 64; ++rep) {
            const uint4 v = random_vec(seed);
            unsigned char vb[16], got[16];
            vec_bytes(v, vb);
            // the whole vector at blk + d
            std::memset(buf, 0xA5, sizeof buf);
            vc::st_aligned<ES>(blk + d, v);
            for (int k = 0; k < 64; ++k) {
                const int rel = k - 16 - d;
                if (buf[k] != ((rel >= 0 && rel < 16) ? vb[rel] : 0xA5)) fail("st_aligned", ES, d, k);
            }
            for (int k = 0; k < 64; ++k) buf[k] = (unsigned char)lcg(seed);
            vec_bytes(vc::ld_aligned<ES>(blk + d), got);
            for (int k = 0; k < 16; ++k)
                if (got[k] != blk[d + k]) fail("ld_aligned", ES, d, k);
            // every element-aligned byte range [from, from + len) of v
            for (int from = 0; from < 16; from += ES) {
                for (int len = ES; from + len <= 16; len += ES) {
                    std::memset(buf, 0xA5, sizeof buf);
                    vc::st_bytes<ES>(blk + d, v, from, len);
                    for (int k = 0; k < 64; ++k) {
                        const int rel = k - 16 - d;  // byte of v stored here, if any
                        const bool in = rel >= 0 && rel < len;
                        if (buf[k] != (in ? vb[from + rel] : 0xA5)) fail("st_bytes", ES, d, k);
                    }
                    for (int k = 0; k < 64; ++k) buf[k] = (unsigned char)lcg(seed);
                    vec_bytes(vc::ld_block_part<ES>(blk, from, from + len), got);
                    for (int k = 0; k < 16; ++k) {
                        const bool in = k >= from && k < from + len;
                        if (got[k] != (in ? blk[k] : 0)) fail("ld_block_part", ES, from, k);
                    }
                }
            }
        }
    }
}

}  // namespace

int main() {
    unsigned seed = 12345u;
    check_es<2>(seed);
    check_es<4>(seed);
    check_es<8>(seed);
    if (failures) {
        std::printf("%d failures\n", failures);
        return 1;
    }
    std::printf("ok\n");
    return 0;
}
