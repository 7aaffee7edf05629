"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, its struct layouts match the Python marshalling, and its
host-side checks (descriptor validator, argument validation) behave.  No call
here launches a kernel."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import position_invariant_kv_chunk_gb300 as K
from position_invariant_kv_chunk_gb300 import build as B

HEADER = os.path.join(B.INCLUDE, "kamera.h")


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:int|size_t|const char\*)\s+(kamera_\w+)\s*\(", src, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kamera_relocate_patch", "kamera_slide_inplace", "kamera_mla_relocate_patch",
              "kamera_ingest_canonical", "kamera_mla_ingest_canonical", "kamera_form_patch",
              "kamera_attend_reused", "kamera_mla_attend_reused", "kamera_validate_chunks", "kamera_status_string",
              "kamera_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = C.CDLL(B.build())
    for n in declared_functions():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    for n in declared_functions():
        assert re.search(rf"\bT {n}$", out, re.M), n


def test_struct_layouts_match_header(tmp_path):
    """Compile a probe against the header with gcc and compare sizes/offsets
    with the ctypes structures the binding marshals."""
    structs = {
        "KameraChunk": K._Chunk, "KameraRope": K._Rope, "KameraGqaPool": K._GqaPool,
        "KameraGqaStore": K._GqaStore, "KameraSlidePool": K._SlidePool, "KameraMlaPool": K._MlaPool,
        "KameraMlaStore": K._MlaStore, "KameraGqaStoreOut": K._GqaStore, "KameraMlaStoreOut": K._MlaStore,
        "KameraDeficit": K._Deficit, "KameraAttnKV": K._AttnKV, "KameraAttnQuery": K._AttnQuery,
        "KameraAttnMlaKV": K._AttnMlaKV,
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kamera.h"', 'int main(void){']
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0;}")
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-I", B.INCLUDE, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {}
    for ln in out:
        if ln:
            s, f, v = ln.split()
            got[(s, f)] = int(v)
    for cname, py in structs.items():
        assert got[(cname, "size")] == C.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)


def test_status_strings_and_version():
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kamera.h")).read()
    declared = int(re.search(r"#define KAMERA_ABI_VERSION (\d+)", hdr).group(1))
    assert K.kamera_abi_version() == declared == K.ABI_VERSION
    for code in range(5):
        assert K.kamera_status_string(code)
    assert K.kamera_status_string(99) == "unknown status"


def _chunk(src, ln, slots, rank=0, delta=0, patches=()):
    return K.ChunkSpec(src, ln, delta, rank, np.asarray(slots, dtype=np.int64), patches)


def test_validator_accepts_disjoint_chunks():
    ch = [_chunk(0, 4, [3, 9, 1, 2]), _chunk(4, 3, [0, 4, 5])]
    assert K.kamera_validate_chunks(ch, 7, 10, 4, 0) == (0, -1, 0)


@pytest.mark.parametrize("mutate,bits,bad", [
    (lambda ch: ch[1].__setattr__("slots", np.array([0, 4, 10])), 1, 1),        # slot == num_slots
    (lambda ch: ch[1].__setattr__("slots", np.array([0, 4, 9])), 1, 1),         # duplicate slot 9
    (lambda ch: ch[0].__setattr__("src_offset", -1), 2, 0),                     # source before the store
    (lambda ch: ch[1].__setattr__("src_offset", 5), 2, 1),                      # source past the store
    (lambda ch: ch[0].__setattr__("length", 5) or ch[0].__setattr__("slots", np.arange(20, 25)), 8, 0),
    (lambda ch: ch[1].__setattr__("rank", 3) or ch[1].__setattr__("patches", (16, 32, 48, 64)), 16, 1),
    (lambda ch: ch[1].__setattr__("rank", 2) or ch[1].__setattr__("patches", (16, 0, 48, 64)), 4, 1),
    (lambda ch: ch[1].__setattr__("rank", 2) or ch[1].__setattr__("patches", (16, 8, 48, 64)), 4, 1),
    (lambda ch: ch[0].__setattr__("delta", 2 ** 40), 4, 0),
])
def test_validator_rejects(mutate, bits, bad):
    ch = [_chunk(0, 4, [3, 9, 1, 2]), _chunk(4, 3, [0, 4, 5])]
    mutate(ch)
    rc, b, got = K.kamera_validate_chunks(ch, 7, 10, 4, 2)
    assert rc == 1 and b == bad and got == bits, (rc, b, got)


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks; run where no GPU exists")
def test_argument_errors_before_any_launch():
    """Each call is malformed, so the library returns before touching CUDA."""
    L, S, H, d = 1, 16, 2, 64
    pk = torch.zeros(L, S, H, d, dtype=torch.bfloat16)
    pv = torch.zeros_like(pk)
    sk = torch.zeros(L, 8, H, d, dtype=torch.bfloat16)
    sv = torch.zeros_like(sk)
    ch = torch.zeros(64, dtype=torch.uint8)
    rope = K.Rope(1e4, 64)
    with pytest.raises(K.KameraError) as e:
        K.kamera_relocate_patch(pk, pv, sk, sv, K.Rope(1e4, 24), ch, 1, 8, 0, stream=0)
    assert e.value.status == 3
    with pytest.raises(K.KameraError) as e:
        K.kamera_relocate_patch(pk, pv, sk, sv, rope, ch, 1, 8, 200, stream=0)
    assert e.value.status == 3
    with pytest.raises(K.KameraError) as e:
        K.kamera_relocate_patch(pk, pv, sk, sv, rope, ch, 1, -8, 0, stream=0)
    assert e.value.status == 1
    with pytest.raises(K.KameraError) as e:
        K.kamera_relocate_patch(pk, pv, torch.as_strided(pk, sk.shape, sk.stride()), sv, rope, ch, 1, 8, 0,
                                stream=0)
    assert e.value.status == 1
    # n_chunks == 0 is a successful no-op that never reaches CUDA
    K.kamera_relocate_patch(pk, pv, sk, sv, rope, ch, 0, 8, 0, stream=0)
    # ingest: overlapping pool and store, a rank-bound call, a no-op
    with pytest.raises(K.KameraError) as e:
        K.kamera_ingest_canonical(pk, pv, torch.as_strided(pk, sk.shape, sk.stride()), sv, rope, ch, 1, 8, stream=0)
    assert e.value.status == 1
    with pytest.raises(K.KameraError) as e:
        K.kamera_ingest_canonical(pk, pv, sk, sv, K.Rope(1e4, 24), ch, 1, 8, stream=0)
    assert e.value.status == 3
    with pytest.raises(K.KameraError) as e:
        K.kamera_ingest_canonical(pk, pv, sk, sv, rope, ch, 1, -1, stream=0)
    assert e.value.status == 1
    K.kamera_ingest_canonical(pk, pv, sk, sv, rope, ch, 0, 8, stream=0)
    mla = torch.zeros(1, 16, 24, dtype=torch.bfloat16)
    with pytest.raises(K.KameraError) as e:
        K.kamera_mla_relocate_patch(mla, torch.zeros(1, 8, 24, dtype=torch.bfloat16), 12,
                                    K.Rope(1e4, 12, 0, K.INTERLEAVED), ch, 1, 8, 0, stream=0)
    assert e.value.status == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks; run where no GPU exists")
def test_form_patch_argument_errors():
    """Malformed patch-formation calls return before touching CUDA."""
    x = torch.zeros(2, 3, 16, 64, dtype=torch.bfloat16)
    for m, status in ((0, 1), (65, 3)):
        with pytest.raises(K.KameraError) as e:
            K.kamera_form_patch(x, m, stream=0)
        assert e.value.status == status
    with pytest.raises(K.KameraError) as e:
        K.kamera_form_patch(torch.zeros(1, 1, 16, 584, dtype=torch.bfloat16), 8, stream=0)   # wider than 576
    assert e.value.status == 3
    with pytest.raises(K.KameraError) as e:
        K.kamera_form_patch(torch.zeros(1, 1, 16, 512, dtype=torch.bfloat16), 33, stream=0)  # wide: rank <= 32
    assert e.value.status == 3
    with pytest.raises(K.KameraError) as e:
        K.kamera_form_patch(torch.zeros(1, 1, 16, 60, dtype=torch.bfloat16), 8, stream=0)    # not a multiple of 8
    assert e.value.status == 3
    with pytest.raises(K.KameraError) as e:
        K.kamera_form_patch(torch.zeros(1, 1, 16, 72, dtype=torch.bfloat16)[..., 4:68], 8, stream=0)   # 8-byte offset
    assert e.value.status == 2
    u = torch.zeros(2, 3, 16, 8, dtype=torch.bfloat16)
    with pytest.raises(K.KameraError) as e:   # u aliases the deficit
        K.kamera_form_patch(torch.as_strided(u, (2, 3, 16, 8), u.stride()), 8, u=u, stream=0)
    assert e.value.status in (1, 3)
    # an empty block grid is a successful no-op
    K.kamera_form_patch(torch.zeros(0, 3, 16, 64, dtype=torch.bfloat16), 8, stream=0)


class _RawRope:
    """A KameraRope built field by field (the binding's own checks bypassed),
    for the library's checks of the multi-axis fields.  The device pointer is
    never dereferenced: each call is malformed and returns before any launch."""

    def __init__(self, n_axes, axes, dptr, rot_dim=64):
        self.n_axes, self.axes, self.dptr, self.rot_dim = n_axes, axes, dptr, rot_dim

    def _c(self, n_chunks=0):
        keep = None
        ap = None
        if self.axes is not None:
            keep = np.ascontiguousarray(self.axes, dtype=np.uint8)
            ap = keep.ctypes.data_as(C.POINTER(C.c_uint8))
        return K._Rope(1e4, self.rot_dim, 0, K.ROTATE_HALF, self.n_axes, None, ap, self.dptr), keep


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks; run where no GPU exists")
def test_axis_rope_argument_errors():
    pk = torch.zeros(1, 16, 2, 64, dtype=torch.bfloat16)
    pv = torch.zeros_like(pk)
    sk = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    sv = torch.zeros_like(sk)
    ch = torch.zeros(64, dtype=torch.uint8)
    fake = 1 << 20   # an 8-byte aligned address that is never read
    axes = np.arange(32) % 3
    for rope, status in ((_RawRope(4, np.zeros(32), fake), 3),            # more than 3 axes
                         (_RawRope(-1, None, None), 1),                    # negative count
                         (_RawRope(2, axes, fake), 1),                     # axis 2 of 2
                         (_RawRope(3, axes, fake + 4), 1),                 # misaligned moves
                         (_RawRope(3, axes, None), 1),                     # no moves
                         (_RawRope(3, None, fake), 1),                     # no axis map
                         (_RawRope(0, axes, None), 1),                     # map without axes
                         (_RawRope(0, None, fake), 1)):                    # moves without axes
        with pytest.raises(K.KameraError) as e:
            K.kamera_relocate_patch(pk, pv, sk, sv, rope, ch, 1, 8, 0, stream=0)
        assert e.value.status == status, (rope.n_axes, status)
        with pytest.raises(K.KameraError) as e:
            K.kamera_slide_inplace(pk, rope, ch, 1, 8, stream=0)
        assert e.value.status == status
    with pytest.raises(ValueError):   # the binding: moves must be a device int64 [n_chunks, n_axes] tensor
        K.Rope(1e4, 64, freq_axis=axes, axis_delta=torch.zeros(1, 3, dtype=torch.int64))._c()
    with pytest.raises(ValueError):
        K.Rope(1e4, 64, freq_axis=axes)._c()


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-only argument checks; run where no GPU exists")
def test_mla_attend_argument_errors():
    """Malformed MLA attention calls return before touching CUDA; no sequences is a no-op."""
    store = torch.zeros(64, 576, dtype=torch.bfloat16)
    q = torch.zeros(2, 16, 576, dtype=torch.bfloat16)
    ch = torch.zeros(64, dtype=torch.uint8)
    seq = torch.zeros(3, dtype=torch.int32)
    rope = K.Rope(1e4, 64, 0, K.INTERLEAVED)
    cases = [
        (dict(q=torch.zeros(2, 129, 576, dtype=torch.bfloat16)), 3),     # more than 128 query heads
        (dict(max_rank=34), 3),                                          # rank above 32
        (dict(store=torch.zeros(64, 320, dtype=torch.bfloat16), kv_lora=256,
              q=torch.zeros(2, 16, 320, dtype=torch.bfloat16)), 3),      # a latent width other than 512
        (dict(store=torch.zeros(64, 580, dtype=torch.bfloat16)[:, :576]), 2),   # row stride not a multiple of 8
        (dict(rope=_RawRope(4, np.zeros(32), 1 << 20)), 3),               # more than 3 RoPE axes
        (dict(max_len=-1), 1),
    ]
    for over, status in cases:
        a = dict(store=store, kv_lora=512, q=q, rope=rope, max_len=8, max_rank=16)
        a.update(over)
        with pytest.raises(K.KameraError) as e:
            K.kamera_mla_attend_reused(a["store"], a["kv_lora"], a["q"], a["rope"], ch, seq, 1, a["max_len"],
                                       a["max_rank"], stream=0)
        assert e.value.status == status, (over, e.value.status)
    out = K.kamera_mla_attend_reused(store, 512, torch.zeros(0, 16, 576, dtype=torch.bfloat16), rope, ch,
                                     torch.zeros(1, dtype=torch.int32), 0, 8, 16, stream=0)
    assert out.shape == (0, 16, 512)


def test_attend_store_row_bound():
    """Attention addresses tile rows with 32-bit coordinates: a store of more
    than 2^31 - 1 rows is UNSUPPORTED, checked before any pointer is used."""
    lib = K.load_library()
    fake = 1 << 20   # never dereferenced: the call returns first
    kv = K._AttnKV(fake, fake, 1 << 31, 128, 2, 64, 0, 0)
    q = K._AttnQuery(fake, fake + (1 << 16), 1, 4, 0.125, 0)
    r, keep = K.Rope(1e4, 64)._c(1)
    rc = lib.kamera_attend_reused(C.byref(kv), C.byref(q), C.byref(r), C.c_void_p(fake), C.c_void_p(fake), 1, 8, 0,
                                  None, 0, None, None)
    assert rc == 3
    kv.num_rows = -1
    assert lib.kamera_attend_reused(C.byref(kv), C.byref(q), C.byref(r), C.c_void_p(fake), C.c_void_p(fake), 1, 8,
                                    0, None, 0, None, None) == 1
    del keep


def test_prefill_argument_errors():
    """Prefill attention's argument checks return before any pointer is used:
    an unsupported head_dim or rank, a store too tall for 32-bit tile rows, a
    negative count, an lse that is not 4-byte aligned, out overlapping q."""
    lib = K.load_library()
    fake = 1 << 20   # never dereferenced: every call returns first
    r, keep = K.Rope(1e4, 64)._c(1)

    def call(kv, q, max_rank=8):
        return lib.kamera_prefill_attend_reused(C.byref(kv), C.byref(q), C.byref(r), C.c_void_p(fake),
                                                C.c_void_p(fake), 1, 8, max_rank, None, None)

    kv = K._AttnKV(fake, fake + (1 << 24), 1024, 128, 2, 64, 0, 0)
    q = K._PrefillQuery(fake + (2 << 24), fake + (3 << 24), fake + (4 << 24), 1, 5, 4, 0.125)
    assert call(kv, q, max_rank=65) == 3                         # ranks up to 64
    kv96 = K._AttnKV(fake, fake + (1 << 24), 1024, 192, 2, 96, 0, 0)
    assert call(kv96, q) == 3                                    # head_dim 64 or 128
    tall = K._AttnKV(fake, fake + (1 << 24), 1 << 31, 128, 2, 64, 0, 0)
    assert call(tall, q) == 3                                    # rows addressed by 32-bit coordinates
    neg = K._PrefillQuery(fake + (2 << 24), fake + (3 << 24), 0, 1, -1, 4, 0.125)
    assert call(kv, neg) == 1
    odd = K._PrefillQuery(fake + (2 << 24), fake + (3 << 24), fake + (4 << 24) + 2, 1, 5, 4, 0.125)
    assert call(kv, odd) == 2                                    # lse 4-byte aligned
    alias = K._PrefillQuery(fake + (2 << 24), fake + (2 << 24), 0, 1, 5, 4, 0.125)
    assert call(kv, alias) == 1                                  # out overlapping q
    empty = K._PrefillQuery(fake + (2 << 24), fake + (3 << 24), 0, 1, 0, 4, 0.125)
    assert call(kv, empty) == 0                                  # no query token: nothing to do
    del keep


def test_compute_calls_take_cuda_tensors_only(monkeypatch):
    """Where CUDA is present, every tensor a compute entry point reads or writes
    must be a CUDA tensor (a host address is not a device address); the binding
    refuses host tensors before anything reaches the library."""
    monkeypatch.setattr(torch.cuda, "is_available", lambda: True)
    pk = torch.zeros(1, 16, 2, 64, dtype=torch.bfloat16)
    sk = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    ch = torch.zeros(64, dtype=torch.uint8)
    rope = K.Rope(1e4, 64)
    calls = [
        lambda: K.kamera_relocate_patch(pk, pk.clone(), sk, sk.clone(), rope, ch, 1, 8, 0, stream=0),
        lambda: K.kamera_slide_inplace(pk, rope, ch, 1, 8, stream=0),
        lambda: K.kamera_ingest_canonical(pk, pk.clone(), sk, sk.clone(), rope, ch, 1, 8, stream=0),
        lambda: K.kamera_form_patch(torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16), 8, stream=0),
        lambda: K.kamera_attend_reused(sk[0], sk[0].clone(), torch.zeros(1, 2, 64, dtype=torch.bfloat16), rope, ch,
                                       torch.zeros(2, dtype=torch.int32), 1, 8, 0, stream=0),
        lambda: K.kamera_mla_attend_reused(torch.zeros(8, 576, dtype=torch.bfloat16), 512,
                                           torch.zeros(1, 16, 576, dtype=torch.bfloat16), K.Rope(1e4, 64), ch,
                                           torch.zeros(2, dtype=torch.int32), 1, 8, 0, stream=0),
        lambda: K.kamera_prefill_attend_reused(sk[0], sk[0].clone(), torch.zeros(1, 3, 2, 64, dtype=torch.bfloat16),
                                               rope, ch, torch.zeros(2, dtype=torch.int32), 1, 8, 0, stream=0),
    ]
    for call in calls:
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
