"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/attnres.h declares, and rejects bad arguments on the host
before any CUDA call is made."""
import ctypes

import pytest

from depth_wise_attention_gb300 import attnres
from depth_wise_attention_gb300.build import build

OK, INV, UNS = attnres.OK, attnres.ERR_INVALID_ARG, attnres.ERR_UNSUPPORTED
F32, BF16 = attnres.F32, attnres.BF16
A = 0x10000           # a fake, 16-byte aligned "device" address (never dereferenced)
B = 0x40000000        # another one, far away


@pytest.fixture(scope="module")
def lib():
    build()
    return attnres.load()


def test_exports_every_declared_function(lib):
    names = attnres.header_functions()
    for must in ("attnres_full_fwd", "attnres_block_phase1", "attnres_block_phase2_merge",
                 "mhar_fwd", "msar_expand_fwd", "attnres_status_string", "attnres_sync_status"):
        assert must in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for s in range(5):
        assert attnres.status_string(s)
    assert attnres.status_string(99) == "unknown status"
    assert "sm_103a" in attnres.version()
    assert attnres.last_cuda_error() == ""


def full(lib, src=A, n_src=8, stride=None, T=16, d=64, dt=BF16, q=B, g=None, eps=1e-6, out=B + 0x100000):
    stride = T * d if stride is None else stride
    return lib.attnres_full_fwd(src, n_src, stride, T, d, dt, q, g, eps, out, None)


def phase1(lib, src=A, n_src=8, stride=None, T=16, d=64, dt=BF16, q=B, n_q=4, g=None, eps=1e-6,
           o=B + 0x100000, lse=B + 0x900000):
    stride = T * d if stride is None else stride
    return lib.attnres_block_phase1(src, n_src, stride, T, d, dt, q, n_q, g, eps, o, lse, None)


def test_full_validation(lib):
    assert full(lib, T=0) == OK                      # empty: no-op, no CUDA call
    assert full(lib, src=None) == INV
    assert full(lib, q=None) == INV
    assert full(lib, out=None) == INV
    assert full(lib, T=-1) == INV
    assert full(lib, n_src=0) == INV
    assert full(lib, d=0) == INV
    assert full(lib, eps=-1.0) == INV
    assert full(lib, eps=float("nan")) == INV
    assert full(lib, eps=float("inf")) == INV
    assert full(lib, stride=16 * 64 - 8) == INV       # sources overlap each other
    assert full(lib, dt=7) == INV
    assert full(lib, out=A + 64) == INV               # output overlaps the sources
    assert full(lib, d=60, stride=16 * 64) == UNS     # d % 8
    assert full(lib, src=A + 8) == UNS                # misaligned source
    assert full(lib, out=B + 0x100008) == UNS         # misaligned output
    assert full(lib, q=B + 4) == UNS                  # misaligned query
    assert full(lib, g=B + 0x200004) == UNS           # misaligned gain
    assert full(lib, stride=16 * 64 + 4, dt=BF16) == UNS   # 8-byte source pitch
    assert full(lib, T=0, src=None, out=None) == OK   # empty: pointers may be NULL
    assert full(lib, T=0, n_src=0) == INV             # scalars are still validated


def test_phase1_and_mhar_validation(lib):
    assert phase1(lib, T=0) == OK
    assert phase1(lib, n_q=0) == INV
    assert phase1(lib, n_q=9) == UNS
    assert phase1(lib, lse=B + 0x900002) == UNS       # lse must be 4-byte aligned
    assert phase1(lib, lse=A) == INV                  # lse overlaps the sources
    assert phase1(lib, o=A + 0x100) == INV
    # MHAR: H must divide d; head width must suit the kernel
    mh = lambda H, d=512, T=0: lib.mhar_fwd(A, 8, T * d, T, d, H, BF16, B, 4, None, 1e-6,
                                            B + 0x100000, None, None)
    assert mh(3) == INV
    assert mh(0) == INV
    assert mh(1) == OK
    assert lib.mhar_fwd(A, 8, 16 * 512, 16, 512, 8, BF16, B, 4, None, 1e-6, B + 0x100000, None,
                        None) == UNS                   # 64-channel heads: not a multiple of 256


def test_phase2_validation(lib):
    m = lambda o=A, lse=B, p=B + 0x100000, T=16, d=64, q=B + 0x200000, out=B + 0x300000, eps=1e-6: \
        lib.attnres_block_phase2_merge(o, lse, p, T, d, BF16, q, None, eps, out, None)
    assert m(T=0) == OK
    assert m(o=None) == INV
    assert m(out=None) == INV
    assert m(lse=None) == INV
    assert m(q=None) == INV
    assert m(o=None, out=None, T=0) == OK
    assert m(out=B + 0x100000 + 16) == INV           # out overlaps partial
    assert m(out=A + 16) == INV                      # out partially overlaps o
    assert m(out=A, T=0) == OK                       # in place is allowed
    assert m(d=12) == UNS
    assert m(p=B + 0x100004) == UNS


def test_phase2_update_and_mhar_phase2_validation(lib):
    P, F, PO, O, L, Q, OUT = A, A + 0x100000, A + 0x200000, B, B + 0x100000, B + 0x200000, B + 0x300000

    def up(p=P, f=F, po=PO, o=O, lse=L, T=16, d=64, q=Q, out=OUT, eps=1e-6):
        return lib.attnres_block_phase2_update_merge(p, f, po, o, lse, T, d, BF16, q, None, eps, out, None)
    assert up(T=0) == OK
    assert up(f=None) == INV                          # the update needs f
    assert up(po=None) == INV                         # ... and somewhere to put p + f
    assert up(lse=None) == INV
    assert up(q=None) == INV
    assert up(po=P, T=0) == OK                        # update in place of the partial
    assert up(po=F, T=0) == OK                        # ... or of f
    assert up(po=P + 16) == INV                       # partially overlapping the partial
    assert up(po=O) == INV                            # the updated partial may not overlap o
    assert up(out=F) == INV                           # out may not overlap f
    assert up(out=PO + 16) == INV                     # ... or the updated partial
    assert up(out=O, T=0) == OK                       # merge in place of o
    assert up(f=F + 8) == UNS                         # misaligned f
    assert up(d=12) == UNS

    def mh(H=8, d=4096, T=16, p=P, f=None, po=None, lse=L):
        return lib.mhar_phase2_merge(O, lse, p, f, po, T, d, H, BF16, Q, None, 1e-6, OUT, None)
    assert mh(T=0) == OK
    assert mh(H=3, T=0) == INV                        # H must divide d
    assert mh(H=0, T=0) == INV
    assert mh(lse=None) == INV
    assert mh(f=F, po=None) == INV                    # an update needs partial_out
    assert mh(H=1, T=0) == OK
    assert mh(H=8, d=4096, T=0) == OK                 # 64 vectors per head
    assert mh(H=16, d=2048, T=0) == OK                # 16 vectors per head (inside a warp)
    assert mh(H=6, d=6 * 40, T=0) == UNS              # 5 vectors per head
    assert mh(H=3, d=3 * 384, T=0) == UNS             # 48 vectors per head


def test_read_bwd_validation(lib):
    SRC, Q, DO, DS, DQ, DG, WS = A, B, B + 0x100000, A + 0x1000000, B + 0x200000, B + 0x300000, B + 0x400000

    def bw(src=SRC, n_src=9, T=16, d=64, q=Q, n_q=1, dout=DO, dsrc=DS, dstride=None, acc=0, dq=DQ, dg=DG,
           ws=WS, wsb=1 << 20, eps=1e-6):
        dstride = T * d if dstride is None else dstride
        return lib.attnres_read_bwd(src, n_src, T * d, T, d, BF16, q, n_q, None, eps, dout, dsrc, dstride, acc,
                                    dq, dg, ws, wsb, None)
    assert bw(n_q=0) == INV
    assert bw(acc=2) == INV
    assert bw(dout=None) == INV
    assert bw(dsrc=None) == INV
    assert bw(dq=None) == INV
    assert bw(ws=None) == INV
    assert bw(dstride=16 * 64 - 8) == INV              # gradient rows of two sources overlap
    assert bw(dsrc=SRC + 64) == INV                    # overlaps the sources
    assert bw(ws=DO + 32) == INV                       # workspace overlaps dout
    assert bw(dq=WS + 64) == INV                       # dq overlaps the workspace
    assert bw(n_src=257) == UNS                        # more than 32 chunks of 8 sources
    assert bw(dout=DO + 8) == UNS                      # misaligned
    assert bw(dg=None, T=0) != INV                     # dgain is optional
    n = ctypes.c_size_t(0)
    assert lib.attnres_read_bwd_workspace_size(9, 16, 64, 1, BF16, None) == INV
    assert lib.attnres_read_bwd_workspace_size(9, 16, 60, 1, BF16, ctypes.byref(n)) == UNS
    assert lib.attnres_read_bwd_workspace_size(257, 16, 64, 1, BF16, ctypes.byref(n)) == UNS
    assert lib.attnres_read_bwd_workspace_size(17, 16, 64, 9, BF16, ctypes.byref(n)) == UNS
    # more queries than one pass takes are accepted (passes of 2, or of 1 above 8 sources)
    for n_src, n_q in ((9, 3), (8, 5)):
        assert lib.attnres_read_bwd_workspace_size(n_src, 16, 64, n_q, BF16, ctypes.byref(n)) not in (INV, UNS)


def test_mhar_read_bwd_validation(lib):
    SRC, Q, DO, DS, DQ, DG, WS = A, B, B + 0x1000000, A + 0x2000000, B + 0x2000000, B + 0x2100000, B + 0x2200000

    def bw(H=8, d=4096, n_src=8, T=16, n_q=2, dt=BF16, dq=DQ, ws=WS):
        return lib.mhar_read_bwd(SRC, n_src, T * d, T, d, H, dt, Q, n_q, None, 1e-6, DO, DS, T * d, 0, dq, DG,
                                 ws, 1 << 20, None)
    assert bw(H=0) == INV
    assert bw(H=3) == INV                              # H must divide d
    assert bw(dq=None) == INV
    assert bw(H=32) == UNS                             # 16 vectors per head: not a multiple of 32
    assert bw(H=3, d=768, T=0) not in (INV, UNS)       # 32 vectors per head: accepted
    n = ctypes.c_size_t(0)
    assert lib.mhar_read_bwd_workspace_size(8, 16, 4096, 3, 2, BF16, ctypes.byref(n)) == INV
    assert lib.mhar_read_bwd_workspace_size(8, 16, 4096, 32, 2, BF16, ctypes.byref(n)) == UNS


def test_msar_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    bad = (ctypes.c_int32 * 3)(4, 0, 12)
    big = (ctypes.c_int32 * 3)(4, 8, 17)

    def ms(m=4, k=ks, T=0, d=256, out=B + 0x100000, mix_eps=1e-6):
        return lib.msar_expand_fwd(A, 8, T * d, T, d, BF16, m, ctypes.cast(k, ctypes.c_void_p),
                                   B, B + 0x200000, None, 1e-6, None, B + 0x300000, mix_eps, out,
                                   None)
    assert ms() == OK
    assert ms(k=bad, T=4) == INV
    assert ms(mix_eps=-1.0) == INV
    assert ms(out=None, T=4) == INV
    assert ms(m=3, T=4) == UNS
    assert ms(k=big, T=4) == UNS

    def mc(t_prev=2, T=0, d=256, stride=None):
        stride = (t_prev + T) * d if stride is None else stride
        return lib.msar_expand_fwd_chunk(A, 8, stride, t_prev, T, d, BF16, 4, ctypes.cast(ks, ctypes.c_void_p),
                                         B, B + 0x200000, None, 1e-6, None, B + 0x300000, 1e-6, B + 0x100000, None)
    assert mc() == OK
    assert mc(t_prev=-1) == INV
    assert mc(t_prev=3, T=4, stride=4 * 256) == INV    # sources hold fewer than t_prev + T rows


def test_msar_two_phase_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    bad = (ctypes.c_int32 * 3)(4, 0, 12)
    kp = lambda k: ctypes.cast(k, ctypes.c_void_p)
    T, d = 16, 256

    def p1(src=A, n_src=8, m=4, k=ks, S=4, o=B + 0x1000000, lse=B + 0x3000000, T=T):
        return lib.msar_block_phase1(src, n_src, T * d, T, d, BF16, m, kp(k), B, B + 0x200000, S, None, 1e-6,
                                     o, lse, None)
    assert p1(T=0) == OK
    assert p1(S=0) == INV
    assert p1(o=None) == INV
    assert p1(k=bad) == INV
    assert p1(o=A + 64) == INV                  # overlaps the sources
    assert p1(m=3) == UNS
    assert p1(n_src=9) == UNS
    assert p1(o=B + 0x1000008) == UNS           # misaligned

    def p2(o=A, lse=B + 0x3000000, part=A + 0x2000000, m=4, k=ks, out=B + 0x1000000, mix_eps=1e-6, T=T):
        return lib.msar_block_phase2(o, lse, part, T, d, BF16, m, kp(k), B, B + 0x200000, None, 1e-6, None,
                                     B + 0x300000, mix_eps, out, None)
    assert p2(T=0) == OK
    assert p2(o=None) == INV
    assert p2(out=None) == INV
    assert p2(mix_eps=-1.0) == INV
    assert p2(k=bad) == INV
    assert p2(out=A + 64) == INV                # overlaps the state
    assert p2(m=3) == UNS
    assert p2(part=A + 0x2000008) == UNS        # misaligned partial


def test_two_phase_backward_validation(lib):
    T, d = 16, 256
    O, L, P, DH, DO, DL, DP, DQ, DG, WS = (A, B, A + 0x100000, A + 0x200000, B + 0x100000, B + 0x300000,
                                           B + 0x200000, B + 0x400000, B + 0x500000, B + 0x600000)

    def p2(o=O, lse=L, part=P, dh=DH, do=DO, dl=DL, dp=DP, acc=0, dq=DQ, dg=DG, ws=WS, T=T, d=d, eps=1e-6):
        return lib.attnres_block_phase2_bwd(o, lse, part, T, d, BF16, B + 0x700000, None, eps, dh, do, dl, dp, acc,
                                            dq, dg, ws, 1 << 20, None)
    assert p2(T=0) not in (INV, UNS)
    assert p2(o=None) == INV
    assert p2(dh=None) == INV
    assert p2(dp=None) == INV                     # a partial needs its gradient buffer
    assert p2(acc=2) == INV
    assert p2(eps=-1.0) == INV
    assert p2(do=DH + 64) == INV                  # d_o overlaps dh
    assert p2(dp=DO + 64) == INV                  # outputs overlap
    assert p2(d=60) == UNS
    assert p2(do=DO + 8) == UNS                   # misaligned
    n = ctypes.c_size_t(0)
    assert lib.attnres_block_phase2_bwd_workspace_size(T, d, BF16, None) == INV
    assert lib.attnres_block_phase2_bwd_workspace_size(T, 60, BF16, ctypes.byref(n)) == UNS

    def p1(dl=DL, dsrc=A + 0x1000000):
        return lib.attnres_block_phase1_bwd(A, 8, T * d, T, d, BF16, B, 4, None, 1e-6, DH, dl, dsrc, T * d, 0,
                                            DQ, DG, WS, 1 << 20, None)
    assert p1(dsrc=None) == INV
    assert p1(dl=A + 0x1000000 + 64) == INV       # d_lse overlaps dsrc
    assert p1(dl=DL + 2) == UNS                   # misaligned d_lse


def test_msar_per_source_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    T, d = 16, 256

    def ps(stride, n_src=8, T=T):
        return lib.msar_expand_fwd_ps(A, n_src, T * d, T, d, BF16, 4, ctypes.cast(ks, ctypes.c_void_p), B, stride,
                                      B + 0x400000, None, 1e-6, None, B + 0x500000, 1e-6, B + 0x600000, None)
    assert ps(0) == INV                           # the per-source entry needs a stride
    assert ps(-1) == INV
    assert ps(d * 24 - 1) == INV                  # sources' kernels would overlap
    assert ps(d * 24, T=0) == OK
    assert ps(1, n_src=1, T=0) == OK              # one source: any positive stride
    assert ps(d * 24 + 2) == UNS                  # kernels not 16-byte aligned


def test_msar_backward_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    bad = (ctypes.c_int32 * 3)(4, 0, 12)
    kp = lambda k: ctypes.cast(k, ctypes.c_void_p)
    T, d = 16, 1024
    DH, DS, DCW, DQ, DG, DMG, DMW, WS = (B + 0x1000000, B + 0x2000000, B + 0x3000000, B + 0x3100000,
                                         B + 0x3200000, B + 0x3300000, B + 0x3400000, B + 0x4000000)

    def mb(n_src=8, T=T, d=d, m=4, k=ks, dh=DH, ds=DS, dstride=None, dcw=DCW, dq=DQ, dg=DG, dmg=DMG, dmw=DMW,
           ws=WS, mix_eps=1e-6):
        dstride = T * d if dstride is None else dstride
        return lib.msar_expand_bwd(A, n_src, T * d, T, d, BF16, m, kp(k), B, B + 0x200000, None, 1e-6, None,
                                   B + 0x300000, mix_eps, dh, ds, dstride, dcw, dq, dg, dmg, dmw, ws, 1 << 30, None)
    assert mb(k=bad) == INV
    assert mb(mix_eps=-1.0) == INV
    assert mb(dh=None) == INV
    assert mb(ds=None) == INV
    assert mb(dq=None) == INV
    assert mb(dmw=None) == INV
    assert mb(ws=None) == INV
    assert mb(dstride=T * d - 1) == INV
    assert mb(ds=A + 64) == INV                   # dsrc overlaps the sources
    assert mb(ws=DH - 64) == INV                  # workspace overlaps dh
    assert mb(dg=DQ + 64) == INV                  # parameter gradients overlap
    assert mb(m=3) == UNS
    assert mb(d=256) == UNS                       # mixer kernels exist for d = 1024, 2048, 4096
    assert mb(n_src=17) == UNS
    assert mb(dmw=DMW + 4) == UNS                 # misaligned projection gradient
    assert mb(dh=DH + 8) == UNS
    n = ctypes.c_size_t(0)
    assert lib.msar_expand_bwd_workspace_size(8, T, d, BF16, 4, kp(ks), None) == INV
    assert lib.msar_expand_bwd_workspace_size(8, T, d, BF16, 4, kp(bad), ctypes.byref(n)) == INV
    assert lib.msar_expand_bwd_workspace_size(8, T, d, BF16, 3, kp(ks), ctypes.byref(n)) == UNS


def test_msar_backward_per_source_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    T, d = 16, 1024
    DH, DS, DCW, DQ, DG, DMG, DMW, WS = (B + 0x1000000, B + 0x2000000, B + 0x3000000, B + 0x3400000,
                                         B + 0x3500000, B + 0x3600000, B + 0x3700000, B + 0x4000000)

    def mp(stride, n_src=8, dcw=DCW):
        return lib.msar_expand_bwd_ps(A, n_src, T * d, T, d, BF16, 4, ctypes.cast(ks, ctypes.c_void_p), B, stride,
                                      B + 0x200000, None, 1e-6, None, B + 0x300000, 1e-6, DH, DS, T * d, dcw, DQ, DG,
                                      DMG, DMW, WS, 1 << 30, None)
    assert mp(0) == INV                           # the per-source entry needs a stride
    assert mp(-4) == INV
    assert mp(d * 24 - 4) == INV                  # sources' kernels would overlap
    assert mp(d * 24, dcw=DQ - 64) == INV         # 8 kernel gradients run into dqueries
    assert mp(d * 24 + 2) == UNS                  # kernels not 16-byte aligned


def test_msar_workspace_chain_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    bad = (ctypes.c_int32 * 3)(4, 0, 12)
    kp = lambda k: ctypes.cast(k, ctypes.c_void_p)
    T, d = 16, 1024
    OUT, WS = B + 0x1000000, B + 0x4000000

    def fw(k=ks, T=T, d=d, cstride=0, out=OUT, ws=WS, mix_eps=1e-6):
        return lib.msar_expand_fwd_ws(A, 8, T * d, T, d, BF16, 4, kp(k), B, cstride, B + 0x200000, None, 1e-6, None,
                                      B + 0x300000, mix_eps, out, ws, 1 << 30, None)
    assert fw(T=0) == OK
    assert fw(k=bad) == INV
    assert fw(mix_eps=-1.0) == INV
    assert fw(out=None) == INV
    assert fw(ws=None) == INV
    assert fw(cstride=-1) == INV
    assert fw(cstride=d * 24 - 1) == INV           # sources' kernels would overlap
    assert fw(out=A + 64) == INV                   # overlaps the sources
    assert fw(ws=OUT - 64) == INV                  # workspace overlaps out
    assert fw(d=1536) == UNS                       # the mixer slices need d % 1024 == 0
    assert fw(out=OUT + 8) == UNS
    n = ctypes.c_size_t(0)
    assert lib.msar_expand_fwd_ws_workspace_size(8, T, d, BF16, None) == INV
    assert lib.msar_expand_fwd_ws_workspace_size(8, T, 1536, BF16, ctypes.byref(n)) == UNS

    def p1(S=4, o=OUT, lse=B + 0x3000000, ws=WS, T=T, d=d):
        return lib.msar_block_phase1_ws(A, 8, T * d, T, d, BF16, 4, kp(ks), B, B + 0x200000, S, None, 1e-6, o, lse,
                                        ws, 1 << 30, None)
    assert p1(T=0) == OK
    assert p1(S=0) == INV
    assert p1(o=None) == INV
    assert p1(ws=None) == INV
    assert p1(o=A + 64) == INV
    assert p1(d=768) == UNS                        # the streams kernel needs d % 512 == 0
    assert lib.msar_block_phase1_ws_workspace_size(8, T, d, BF16, 0, ctypes.byref(n)) == INV


def test_msar_phase2_workspace_chain_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    T, d = 16, 1024

    def p2(o=A, part=A + 0x2000000, out=B + 0x1000000, ws=B + 0x4000000, d=d, mix_eps=1e-6):
        return lib.msar_block_phase2_ws(o, B + 0x3000000, part, T, d, BF16, 4, ctypes.cast(ks, ctypes.c_void_p), B,
                                        B + 0x200000, None, 1e-6, None, B + 0x300000, mix_eps, out, ws, 1 << 30, None)
    assert p2(o=None) == INV
    assert p2(ws=None) == INV
    assert p2(mix_eps=-1.0) == INV
    assert p2(out=A + 64) == INV                   # overlaps the state
    assert p2(ws=A + 0x2000000 - 64) == INV        # workspace overlaps the partial
    assert p2(d=1536) == UNS
    n = ctypes.c_size_t(0)
    assert lib.msar_block_phase2_ws_workspace_size(T, 1536, BF16, ctypes.byref(n)) == UNS


def test_msar_two_phase_backward_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    bad = (ctypes.c_int32 * 3)(4, 0, 12)
    kp = lambda k: ctypes.cast(k, ctypes.c_void_p)
    T, d = 16, 1024
    O, L, P, DH = A, B, A + 0x1000000, A + 0x2000000
    DO, DL, DP, WS = B + 0x1000000, B + 0x2000000, B + 0x3000000, B + 0x8000000
    DCW, DQ, DG, DMG, DMW = B + 0x4000000, B + 0x4100000, B + 0x4200000, B + 0x4300000, B + 0x4400000

    def p2(k=ks, part=P, do=DO, dl=DL, dp=DP, ws=WS, d=d, mix_eps=1e-6):
        return lib.msar_block_phase2_bwd(O, L, part, T, d, BF16, 4, kp(k), B + 0x500000, B + 0x600000, None, 1e-6,
                                         None, B + 0x700000, mix_eps, DH, do, dl, dp, DCW, DQ, DG, DMG, DMW, ws,
                                         1 << 30, None)
    assert p2(k=bad) == INV
    assert p2(mix_eps=-1.0) == INV
    assert p2(do=None) == INV
    assert p2(dp=None) == INV                      # a partial needs its gradient buffer
    assert p2(ws=None) == INV
    assert p2(do=O + 64) == INV                    # d_o overlaps the state
    assert p2(dp=DO + 64) == INV                   # outputs overlap
    assert p2(d=1536) == UNS
    assert p2(do=DO + 8) == UNS

    def p1(k=ks, dsrc=B + 0x5000000, ws=WS, d=d, S=4):
        return lib.msar_block_phase1_bwd(A, 8, T * d, T, d, BF16, 4, kp(k), B + 0x500000, B + 0x600000, S, None,
                                         1e-6, DO, DL, dsrc, T * d, DCW, DQ, DG, ws, 1 << 30, None)
    assert p1(k=bad) == INV
    assert p1(S=0) == INV
    assert p1(dsrc=None) == INV
    assert p1(dsrc=A + 64) == INV                  # dsrc overlaps the sources
    assert p1(ws=DO - 64) == INV                   # workspace overlaps d_o
    assert p1(d=768) == UNS


def test_read_bwd_noalloc_validation(lib):
    """The no-allocation backward sizes its passes with attnres_read_bwd's
    workspace rules first, so those rejections come before the device is
    touched."""
    SRC, Q, DO, DS, DQ, DG = A, B, B + 0x100000, A + 0x1000000, B + 0x200000, B + 0x300000

    def na(n_src=9, T=16, d=64, n_q=1, dt=BF16):
        return lib.attnres_read_bwd_noalloc(SRC, n_src, T * d, T, d, dt, Q, n_q, None, 1e-6, DO, DS, T * d, 0,
                                            DQ, DG, None)
    assert na(n_q=0) == INV
    assert na(dt=7) == INV
    assert na(d=60) == UNS                           # rows not a whole number of 16-byte vectors
    assert na(n_src=257) == UNS                      # more than 32 chunks of 8 sources
    assert na(n_src=17, n_q=9) == UNS                # more than 8 queries over more than 16 sources


def test_msar_backward_chunk_validation(lib):
    """The chunked MSAR backward: history rows widen every source and source-
    gradient extent, and T_prev / accumulate have their own checks."""
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    bad = (ctypes.c_int32 * 3)(4, 0, 12)
    kp = lambda k: ctypes.cast(k, ctypes.c_void_p)
    T, d, H = 16, 1024, 11
    DH, DS, DCW, DQ, DG, DMG, DMW, WS = (B + 0x1000000, B + 0x2000000, B + 0x3000000, B + 0x3100000,
                                         B + 0x3200000, B + 0x3300000, B + 0x3400000, B + 0x4000000)

    def mc(t_prev=H, n_src=8, T=T, d=d, k=ks, sstride=None, ds=DS, dstride=None, acc=0, dh=DH, ws=WS):
        rows = t_prev + T if t_prev >= 0 else T
        sstride = rows * d if sstride is None else sstride
        dstride = rows * d if dstride is None else dstride
        return lib.msar_expand_bwd_chunk(A, n_src, sstride, t_prev, T, d, BF16, 4, kp(k), B, B + 0x200000, None,
                                         1e-6, None, B + 0x300000, 1e-6, dh, ds, dstride, acc, DCW, DQ, DG, DMG,
                                         DMW, ws, 1 << 30, None)
    assert mc(t_prev=-1) == INV
    assert mc(acc=2) == INV
    assert mc(acc=-1) == INV
    assert mc(k=bad) == INV
    assert mc(sstride=T * d) == INV                  # the history rows would overlap the next source
    assert mc(dstride=(H + T) * d - 1) == INV        # so would the gradient rows
    assert mc(ds=A + 64) == INV                      # dsrc overlaps the sources' history rows
    assert mc(ws=DS + 64) == INV                     # workspace overlaps dsrc
    assert mc(d=256) == UNS
    assert mc(n_src=17) == UNS
    assert mc(dh=DH + 8) == UNS
    # T_prev = 0 is the plain backward's argument set; both pass the host checks
    assert mc(t_prev=0) not in (INV, UNS)
    assert mc() not in (INV, UNS)


def test_msar_two_phase_backward_workspace_size_validation(lib):
    ks = (ctypes.c_int32 * 3)(4, 8, 12)
    bad = (ctypes.c_int32 * 3)(4, 0, 12)
    kp = lambda k: ctypes.cast(k, ctypes.c_void_p)
    n = ctypes.c_size_t(0)
    p2 = lambda T=16, d=1024, dt=BF16, m=4, k=ks, out=ctypes.byref(n): \
        lib.msar_block_phase2_bwd_workspace_size(T, d, dt, m, kp(k), out)
    p1 = lambda n_src=8, T=16, d=1024, dt=BF16, m=4, k=ks, S=4, out=ctypes.byref(n): \
        lib.msar_block_phase1_bwd_workspace_size(n_src, T, d, dt, m, kp(k), S, out)
    for f in (p1, p2):
        assert f(out=None) == INV
        assert f(dt=7) == INV
        assert f(T=-1) == INV
        assert f(d=0) == INV
        assert f(k=bad) == INV
        assert f(m=3) == UNS
    assert p1(n_src=0) == INV
    assert p1(S=0) == INV


def test_binding_covers_every_entry_point_and_fails_loudly_without_the_library(tmp_path):
    """The ctypes binding declares a signature for exactly the functions the
    header declares, and with no library there is an error, never a fallback."""
    from depth_wise_attention_gb300 import attnres
    assert set(attnres.header_functions()) == set(attnres._SIGS)
    saved = attnres._lib
    attnres._lib = None
    try:
        with pytest.raises(RuntimeError):
            attnres.load(str(tmp_path / "libattnres.so"))
    finally:
        attnres._lib = saved
