// Host-only dump of the INT2 ledger index maps the CUDA kernels use
// (LedgerLayout in csrc/kvev_internal.h), one line per entry, so a CPU test
// can compare them with the tests' own statement of the layout.
#include <cstdio>

#include "../decoding_kv_cache_split_gb300/csrc/kvev_internal.h"

int main() {
    using L = kvev::LedgerLayout<128>;
    std::printf("offsets %d %d %d %d %d %d %d\n", L::KC, L::KS, L::KZ, L::VC, L::VS, L::VZ, L::BYTES);
    for (int tok = 0; tok < 128; ++tok)
        for (int c = 0; c < 128; ++c) {
            int w, reg, e;
            L::key_place(tok, c, &w, &reg, &e);   // reg: the key's field
            std::printf("k %d %d %d %d %d\n", tok, c, w, reg, L::key_bit(reg, e));
            L::value_place(tok, c, &w, &reg, &e);
            std::printf("v %d %d %d %d %d\n", tok, c, w, L::sign_bit(reg, e), L::mag_bit(reg, e));
        }
    for (int grp = 0; grp < 4; ++grp)
        for (int c = 0; c < 128; ++c) std::printf("ks %d %d %d\n", grp, c, L::key_scale_index(grp, c));
    for (int tok = 0; tok < 128; ++tok)
        for (int cg = 0; cg < 4; ++cg)
            std::printf("vs %d %d %d\n", tok, cg, L::value_scale_index(tok, cg));
    for (unsigned c = 0; c < 4; ++c)
        std::printf("code %u %u %u %u\n", c, kvev::code_sign(c), kvev::code_mag(c),
                    kvev::code_from_bits(kvev::code_sign(c), kvev::code_mag(c)));
    return 0;
}
