// fused.cu -- host side of the one-kernel layer step: the shared-memory plan
// and the table of compiled instances (fused_inst_*.cu).
#include <algorithm>

#include "fused.cuh"

namespace gattn {


bool fused_plan(FusedArgs &a, int num_sms, int max_smem)
{
    if (num_sms + 1 > kFMaxContrib || a.d % 64 || a.d > 256 || a.d == 192)
        return false;
    const long long Ta = (long long)a.nrb_a * a.nku_a;
    const long long per = (Ta + num_sms - 1) / num_sms;
    const long long To = (long long)a.nrb_o * a.nku_o;
    const long long per_o = (To + num_sms - 1) / num_sms;
    if (per_o > 64)                     // row-block arrivals of one CTA fit a 64-bit mask
        return false;
    // q|k|v operand slots, later the o_proj operand of this CTA's k units
    a.xslots = (int)std::max(std::min<long long>(a.nku_a, std::max<long long>(per, 1)),
                             std::min<long long>(a.nku_o, per_o + 1));
    a.xslot_bytes = kXSlotBytes;
    const int DB = a.d / 64;
    const int attn_u = a.MT * 16 * a.d * 2 + a.MT * 16 * 128;
    int u = std::max(attn_u, kMergeBytes);
    u = (u + 127) & ~127;
    const int xbytes = (a.xslots * kXSlotBytes + 127) & ~127;
    const int fixed = xbytes + u + kRedBytes + kStgBytes + kKvnBytes + kMiscBytes + 1024;
    const int ring = (max_smem - fixed) & ~1023;
    const int need = std::max(std::max(round1k(a.step_a), kv_entry_bytes(DB, 3)),
                              std::max(o_entry_bytes(a.step_o),
                                       x_entry_bytes(a.M, a.xslots, a.x_f32 ? 4 : 2)));
    if (ring < 2 * need)
        return false;
    a.ring_bytes = ring;
    a.off_x = ring;
    a.off_u = ring + xbytes;
    a.off_red = a.off_u + u;
    a.off_misc = a.off_red + kRedBytes + kStgBytes + kKvnBytes;
    a.smem_bytes = a.off_misc + kMiscBytes + 1024;
    return a.smem_bytes <= max_smem;
}

bool fused_ops_part1(const FusedKey &k, FusedOps *ops);
bool fused_ops_part2(const FusedKey &k, FusedOps *ops);
bool fused_ops_part3(const FusedKey &k, FusedOps *ops);

bool fused_ops(const FusedKey &k, FusedOps *ops)
{
    return fused_ops_part1(k, ops) || fused_ops_part2(k, ops) || fused_ops_part3(k, ops);
}

}  // namespace gattn
