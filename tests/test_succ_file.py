"""Successor-table files (gt_succ_save / gt_succ_file_shape / gt_succ_load) on the host: the
round trip, the header fields and checksums read independently (struct and zlib), and every
kind of damaged or mismatched file refused with the table left as it was."""
import struct
import zlib

import numpy as np
import pytest


@pytest.fixture(scope="module")
def gt():
    from tree_speculative_decoding_parent_gb300 import build, gt
    build.build()
    return gt


def _table(V, k, seed=0):
    rng = np.random.default_rng(seed)
    t = rng.integers(-1, V, size=(V, k)).astype(np.int32)
    t[0, :] = -1          # an empty row
    t[-1, :] = V - 1      # the largest id
    return t


def test_crc32_definition_check_value(gt, tmp_path):
    """The payload checksum is the standard CRC-32 (check value 0xCBF43926 over "123456789",
    as zlib computes it): the stored value equals zlib's CRC-32 of the table's
    little-endian bytes."""
    assert zlib.crc32(b"123456789") == 0xCBF43926
    t = _table(300, 8, 1)
    p = tmp_path / "t.succ"
    gt.gt_succ_save(str(p), t)
    raw = p.read_bytes()
    assert struct.unpack_from("<I", raw, 24)[0] == zlib.crc32(t.astype("<i4").tobytes())


def test_round_trip_and_header(gt, tmp_path):
    for V, k in ((1, 1), (32000, 8), (151936, 8), (17, 16)):
        t = _table(V, k, V)
        p = tmp_path / f"t{V}.succ"
        gt.gt_succ_save(str(p), t)
        raw = p.read_bytes()
        assert raw[:8] == b"GTSUCC\x00\x01"
        fv, fk, nbytes, crc, hcrc = struct.unpack_from("<IIQII", raw, 8)
        assert (fv, fk, nbytes) == (V, k, 4 * V * k) and len(raw) == 32 + 4 * V * k
        assert hcrc == zlib.crc32(raw[:28])
        assert gt.gt_succ_file_shape(str(p)) == (V, k)
        assert np.array_equal(gt.gt_succ_load(str(p), V, k), t)
        assert np.array_equal(np.frombuffer(raw[32:], "<i4").reshape(V, k), t)
        assert not (tmp_path / f"t{V}.succ.tmp").exists()


def _load_status(gt, path, V, k):
    so = gt.load()
    t = np.full((V, k), 12345, np.int32)
    rc = so.gt_succ_load(str(path).encode(), t.ctypes.data, V, k)
    return rc, bool((t == 12345).all())


def test_damaged_files_are_refused_and_the_table_is_untouched(gt, tmp_path):
    V, k = 1000, 8
    p = tmp_path / "good.succ"
    gt.gt_succ_save(str(p), _table(V, k, 3))
    raw = bytearray(p.read_bytes())
    cases = {}
    b = bytearray(raw); b[32 + 4 * 123] ^= 0x01; cases["payload bit"] = (b, gt.GT_ERR_CORRUPT)
    b = bytearray(raw); b[9] ^= 0x01; cases["header bit"] = (b, gt.GT_ERR_CORRUPT)
    b = bytearray(raw); b[0:1] = b"X"; cases["magic"] = (b, gt.GT_ERR_CORRUPT)
    b = bytearray(raw); b[24] ^= 0xFF; cases["stored payload crc"] = (b, gt.GT_ERR_CORRUPT)
    cases["truncated payload"] = (raw[:-4], gt.GT_ERR_IO)
    cases["truncated header"] = (raw[:20], gt.GT_ERR_IO)
    cases["trailing byte"] = (raw + b"\x00", gt.GT_ERR_IO)
    # a well-formed file (both checksums right) holding an id >= V
    body = bytearray(raw[32:]); struct.pack_into("<i", body, 0, V)
    hdr = bytearray(raw[:32]); struct.pack_into("<I", hdr, 24, zlib.crc32(bytes(body)))
    struct.pack_into("<I", hdr, 28, zlib.crc32(bytes(hdr[:28])))
    cases["id out of range"] = (hdr + body, gt.GT_ERR_CORRUPT)
    for name, (data, want) in cases.items():
        q = tmp_path / "bad.succ"
        q.write_bytes(bytes(data))
        rc, untouched = _load_status(gt, q, V, k)
        assert rc == want, name
        assert untouched, name
    rc, untouched = _load_status(gt, p, V + 1, k)
    assert rc == gt.GT_ERR_SHAPE and untouched
    rc, untouched = _load_status(gt, p, V, k - 1)
    assert rc == gt.GT_ERR_SHAPE and untouched
    rc, untouched = _load_status(gt, tmp_path / "missing.succ", V, k)
    assert rc == gt.GT_ERR_IO and untouched
    rc, _ = _load_status(gt, p, V, k)
    assert rc == gt.GT_OK


def test_save_refuses_out_of_range_entries(gt, tmp_path):
    so = gt.load()
    for bad in (-2, 50):
        t = _table(50, 4)
        t[7, 2] = bad
        p = tmp_path / "x.succ"
        assert so.gt_succ_save(str(p).encode(), t.ctypes.data, 50, 4) == gt.GT_ERR_ARG
        assert not p.exists()
    assert so.gt_succ_save(None, t.ctypes.data, 50, 4) == gt.GT_ERR_ARG
    assert so.gt_succ_save(str(tmp_path / "no_dir" / "x.succ").encode(),
                           _table(50, 4).ctypes.data, 50, 4) == gt.GT_ERR_IO
