"""Host-only checks of the C ABI (no GPU needed, no kernel is launched).

The library is built with nvcc (cross-compiling for sm_103a works without a
GPU); these tests load it, check that it exports every function include/gdn.h
declares, that the ctypes mirrors of the ABI structs match the C layout, and
that invalid arguments are rejected on the host with the documented codes
before any CUDA call is made.
"""
import ctypes as C
import os
import subprocess

import pytest

from hybrid_ssm_gated_gb300 import build, gdn

FAKE = 0x7F0000000000  # 16-byte aligned stand-in pointer; never dereferenced on these paths


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gdn.lib()


def test_exports_every_declared_symbol(lib):
    names = gdn.declared_symbols()
    assert set(names) >= {"gdn_decode_step", "gdn_replay_step", "gdn_replay_flush", "gdn_verify_window",
                          "gdn_rollback", "gdn_last_error_string", "gdn_abi_version", "gdn_spec_step",
                          "mamba2_decode_step", "mamba2_replay_step", "mamba2_verify_window", "mamba2_replay_flush",
                          "mamba2_rollback"}
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/gdn.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_abi_version(lib):
    assert gdn.gdn_abi_version() == 4


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gdn.h"\nint main(void){'
                   'printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(gdn_dims), offsetof(gdn_dims, num_slots),'
                   'sizeof(gdn_replay_cache), offsetof(gdn_replay_cache, ring_rec),'
                   'offsetof(gdn_replay_cache, ckpt_pos), offsetof(gdn_replay_cache, L),'
                   'offsetof(gdn_replay_cache, ckpt_read), offsetof(gdn_replay_cache, read_dtype));'
                   'printf("%zu %zu %zu\\n", sizeof(mamba2_dims), offsetof(mamba2_dims, P),'
                   'offsetof(mamba2_dims, num_slots)); return 0;}\n')
    exe = tmp_path / "layout"
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run(["gcc", "-std=c11", "-I", inc, str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    want = [C.sizeof(gdn.gdn_dims), gdn.gdn_dims.num_slots.offset, C.sizeof(gdn.gdn_replay_cache),
            gdn.gdn_replay_cache.ring_rec.offset, gdn.gdn_replay_cache.ckpt_pos.offset,
            gdn.gdn_replay_cache.L.offset, gdn.gdn_replay_cache.ckpt_read.offset,
            gdn.gdn_replay_cache.read_dtype.offset, C.sizeof(gdn.mamba2_dims), gdn.mamba2_dims.P.offset,
            gdn.mamba2_dims.num_slots.offset]
    assert got == want


def _dims(B=4, Hk=2, Hv=4, dk=128, dv=128, num_slots=8):
    return gdn.gdn_dims(B, Hk, Hv, dk, dv, num_slots)


def _decode(lib, dims, pool=FAKE, sdt=0, slots=FAKE, q=FAKE, k=FAKE, v=FAKE, a=FAKE, b=FAKE, idt=1, A=FAKE,
            dt=FAKE, out=FAKE, odt=0, err=FAKE):
    d = C.byref(dims) if dims is not None else None
    return lib.gdn_decode_step(d, pool, sdt, slots, q, k, v, a, b, idt, A, dt, out, odt, err, None)


def _cache(L=16, ckpt=FAKE, cdt=0, rdt=1, read=None, read_dt=0):
    return gdn.gdn_replay_cache(ckpt, cdt, FAKE, FAKE, rdt, FAKE, FAKE, FAKE, L, read, read_dt)


def test_decode_rejections(lib):
    assert _decode(lib, None) == -1  # GDN_ERR_NULL
    assert "dims" in gdn.gdn_last_error_string()
    assert _decode(lib, _dims(dk=96)) == -3  # GDN_ERR_SHAPE
    assert _decode(lib, _dims(dv=8)) == -3
    assert _decode(lib, _dims(dv=264)) == -3
    assert _decode(lib, _dims(dv=40)) == -3
    assert _decode(lib, _dims(Hk=3, Hv=4)) == -3
    assert _decode(lib, _dims(B=-1)) == -3
    assert _decode(lib, _dims(), pool=None) == -1
    assert _decode(lib, _dims(), err=None) == -1
    assert _decode(lib, _dims(), q=None) == -1
    assert _decode(lib, _dims(), sdt=3) == -2  # GDN_ERR_DTYPE
    assert _decode(lib, _dims(), idt=7) == -2
    assert _decode(lib, _dims(), odt=-1) == -2
    assert _decode(lib, _dims(), q=FAKE + 8) == -5  # GDN_ERR_ALIGN
    assert _decode(lib, _dims(), pool=FAKE + 4) == -5
    assert _decode(lib, _dims(), out=FAKE + 2) == -5
    assert "align" in gdn.gdn_last_error_string()


def test_empty_batch_launches_nothing(lib):
    # B == 0 returns before touching any pointer or the CUDA runtime
    assert _decode(lib, _dims(B=0), pool=None, slots=None) == 0
    d, c = _dims(B=0), _cache()
    assert lib.gdn_replay_step(C.byref(d), C.byref(c), None, None, None, None, None, None, 1, None, None, None, 0,
                               None, None) == 0
    assert lib.gdn_rollback(C.byref(d), C.byref(c), None, None, 4, None, None) == 0


def _verify(lib, dims, cache, T, idt=1):
    return lib.gdn_verify_window(C.byref(dims), C.byref(cache), FAKE, T, FAKE, FAKE, FAKE, FAKE, FAKE, idt, FAKE,
                                 FAKE, FAKE, 0, FAKE, None)


def test_replay_rejections(lib):
    d = _dims()
    assert _verify(lib, d, _cache(L=16), 0) == -4  # GDN_ERR_WINDOW: T < 1
    assert _verify(lib, d, _cache(L=4), 5) == -4  # T > L
    assert _verify(lib, d, _cache(L=16), 9) == -4  # T > 8
    assert _verify(lib, d, _cache(L=65), 4) == -4  # L > 64
    assert lib.gdn_rollback(C.byref(d), C.byref(_cache(L=65)), FAKE, FAKE, 4, FAKE, None) == -4
    assert _verify(lib, d, _cache(L=0), 1) == -4
    assert _verify(lib, d, _cache(rdt=0), 4, idt=1) == -2  # input dtype differs from the ring's
    assert _verify(lib, d, _cache(cdt=5), 4) == -2
    assert _verify(lib, d, _cache(ckpt=FAKE + 8), 4) == -5
    assert _verify(lib, d, _cache(ckpt=None), 4) == -1
    assert lib.gdn_replay_step(C.byref(d), None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 0, FAKE,
                               None) == -1
    assert lib.gdn_replay_flush(C.byref(_dims(dk=48)), C.byref(_cache()), FAKE, 1, FAKE, None) == -3
    assert _verify(lib, _dims(dv=48), _cache(), 4) == -3  # replay needs dv % 32 == 0
    assert lib.gdn_rollback(C.byref(d), C.byref(_cache(L=4)), FAKE, FAKE, 5, FAKE, None) == -4
    assert lib.gdn_rollback(C.byref(d), C.byref(_cache()), FAKE, None, 4, FAKE, None) == -1
    # a read copy needs an fp32 checkpoint and a bf16/fp16 copy, 16-byte aligned
    assert _verify(lib, d, _cache(read=FAKE, read_dt=0), 4) == -2
    assert _verify(lib, d, _cache(cdt=1, read=FAKE, read_dt=1), 4) == -2
    assert _verify(lib, d, _cache(read=FAKE + 8, read_dt=1), 4) == -5


def test_binding_refuses_host_tensors(lib):
    import torch

    t = torch.zeros(4)
    with pytest.raises(ValueError):
        gdn._ptr(t)


def _spec(lib, dims, T=4, pool=FAKE, sdt=0, src=FAKE, dst=FAKE, q=FAKE, idt=1, err=FAKE):
    return lib.gdn_spec_step(C.byref(dims), pool, sdt, src, dst, T, q, FAKE, FAKE, FAKE, FAKE, idt, FAKE, FAKE,
                             FAKE, 0, err, None)


def test_spec_rejections(lib):
    d = _dims()
    assert _spec(lib, d, T=0) == -4  # GDN_ERR_WINDOW
    assert _spec(lib, d, T=9) == -4
    assert _spec(lib, _dims(dk=96)) == -3
    assert _spec(lib, d, dst=None) == -1
    assert _spec(lib, d, err=None) == -1
    assert _spec(lib, d, sdt=4) == -2
    assert _spec(lib, d, idt=5) == -2
    assert _spec(lib, d, pool=FAKE + 8) == -5
    assert _spec(lib, d, q=FAKE + 4) == -5
    assert _spec(lib, _dims(B=0), pool=None, src=None, dst=None) == 0  # nothing to do, nothing touched


def _m2dims(B=4, G=2, H=8, N=128, P=64, num_slots=8):
    return gdn.mamba2_dims(B, G, H, N, P, num_slots)


def _m2decode(lib, dims, pool=FAKE, sdt=0, x=FAKE, dt=FAKE, Bm=FAKE, Cm=FAKE, idt=1, D=FAKE, err=FAKE):
    d = C.byref(dims) if dims is not None else None
    return lib.mamba2_decode_step(d, pool, sdt, FAKE, x, dt, Bm, Cm, idt, FAKE, FAKE, D, FAKE, 0, err, None)


def _m2verify(lib, dims, cache, T, D=FAKE, idt=1):
    return lib.mamba2_verify_window(C.byref(dims), C.byref(cache), FAKE, T, FAKE, FAKE, FAKE, FAKE, idt, FAKE,
                                    FAKE, D, FAKE, 0, FAKE, None)


def test_mamba2_rejections(lib):
    assert _m2decode(lib, None) == -1
    assert _m2decode(lib, _m2dims(N=96)) == -3  # state dim not in {32, 64, 128}
    assert _m2decode(lib, _m2dims(P=40)) == -3
    assert _m2decode(lib, _m2dims(G=3, H=8)) == -3  # H not a multiple of G
    assert _m2decode(lib, _m2dims(), D=None) == -1
    assert _m2decode(lib, _m2dims(), dt=None) == -1
    assert _m2decode(lib, _m2dims(), Cm=FAKE + 4) == -5
    assert _m2decode(lib, _m2dims(), sdt=3) == -2
    assert _m2decode(lib, _m2dims(B=0), pool=None) == 0
    d = _m2dims()
    assert _m2verify(lib, d, _cache(), 4, D=None) == -1
    assert _m2verify(lib, d, _cache(), 4, D=FAKE + 2) == -5
    assert _m2verify(lib, d, _cache(L=4), 5) == -4
    assert _m2verify(lib, d, _cache(), 0) == -4
    assert _m2verify(lib, _m2dims(P=48), _cache(), 4) == -3  # replay needs P % 32 == 0
    assert _m2verify(lib, d, _cache(read=FAKE, read_dt=1), 4) == -2  # no read copy for Mamba2
    assert "Mamba2" in gdn.gdn_last_error_string()
    assert lib.mamba2_replay_step(C.byref(d), C.byref(_cache(rdt=0)), FAKE, FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE,
                                  FAKE, FAKE, 0, FAKE, None) == -2  # input dtype differs from the ring's
    assert lib.mamba2_replay_flush(C.byref(_m2dims(N=48)), C.byref(_cache()), FAKE, 1, FAKE, None) == -3
    assert lib.mamba2_rollback(C.byref(d), C.byref(_cache(L=4)), FAKE, FAKE, 5, FAKE, None) == -4
    assert lib.mamba2_rollback(C.byref(_m2dims(B=0)), C.byref(_cache()), None, None, 4, None, None) == 0


def _prefill(lib, dims, interval=64, total=32, pool=FAKE, cu=FAKE, q=FAKE, b=FAKE, idt=1, err=FAKE, out=FAKE):
    return lib.gdn_prefill(C.byref(dims), pool, 0, FAKE, cu, total, q, FAKE, FAKE, FAKE, b, idt, FAKE, FAKE, interval,
                           out, 0, err, None)


def test_prefill_rejections(lib):
    d = _dims()
    assert _prefill(lib, d, interval=0) == -4  # GDN_ERR_WINDOW
    assert _prefill(lib, d, total=-1) == -3
    assert _prefill(lib, _dims(dk=96)) == -3
    assert _prefill(lib, d, cu=None) == -1
    assert _prefill(lib, d, b=None) == -1
    assert _prefill(lib, d, err=None) == -1
    assert _prefill(lib, d, idt=9) == -2
    assert _prefill(lib, d, q=FAKE + 4) == -5
    assert _prefill(lib, d, pool=FAKE + 8) == -5
    assert _prefill(lib, d, out=FAKE + 8) == -5  # outputs leave in 16-byte vectors
    assert _prefill(lib, d, total=1 << 30) == -3  # total_tokens * Hv too large
    assert _prefill(lib, _dims(B=0), pool=None, cu=None) == 0
