"""Test-side readers of the cache formats documented in include/qevict.h.

These decode the fragment-native bf16 blocks and code fields from their documented formulas,
independently of the CUDA sources, so GPU state can be compared with the oracle.
"""
import numpy as np

D = 128


def _maps(W):
    tok = np.repeat(np.arange(W), D)
    dim = np.tile(np.arange(D), W)
    return tok, dim


def _frag(r, c):
    lane = (r % 8) * 4 + (c % 8) // 2
    reg = r // 8 + 2 * (c // 8)
    return lane, reg


def fn_index(W, is_v):
    """Element index of (tok, dim) inside a fragment-native block, as a [W][D] array."""
    tok, dim = _maps(W)
    r, c = (dim % 16, tok % 16) if is_v else (tok % 16, dim % 16)
    lane, reg = _frag(r, c)
    grp = (tok // 16) * 8 + dim // 16
    return ((grp * 32 + lane) * 8 + reg * 2 + c % 2).reshape(W, D)


def code_position(W, bits, is_v):
    """(byte offset, bit shift) of every (tok, dim) code inside a K or V code block."""
    assert bits in (2, 4)
    tok, dim = _maps(W)
    if bits == 4:
        r, c = (dim % 16, tok % 16) if is_v else (tok % 16, dim % 16)
        lane, reg = _frag(r, c)
        tile = (tok // 16) * 8 + dim // 16
        word = ((tile // 4) * 32 + lane) * 4 + tile % 4
        bit = 4 * reg + 16 * (tok % 2) if is_v else 4 * (reg * 2 + dim % 2)
        return (word * 4 + bit // 8).reshape(W, D), (bit % 8).reshape(W, D)
    if not is_v:
        r, c = tok % 16, dim % 16
        lane, reg = _frag(r, c)
        grp = (tok // 16) * 8 + dim // 16
        e = reg * 2 + c % 2
        bit = np.where(e < 4, 4 * e, 4 * (e - 4) + 2)
        lb = grp * 2 + bit // 8
    else:
        r, c = dim % 16, tok % 16
        lane, _ = _frag(r, c)
        i = dim // 16                        # word i of the lane's 32 bytes
        tau = 2 * (tok // 16) + c // 8       # token pair of the A register
        bit = 8 * (r // 8) + 2 * tau + 16 * (c % 2)
        lb = 4 * i + bit // 8
    byte = (lb // 16) * 512 + lane * 16 + lb % 16
    return byte.reshape(W, D), (bit % 8).reshape(W, D)


def bf16_bits_to_f32(u16):
    return (np.asarray(u16, np.uint32) << 16).view(np.float32)


def unpack_block(block_u16, W, is_v):
    """[W*D] uint16 fragment-native block -> [W][D] float32 values."""
    return bf16_bits_to_f32(np.asarray(block_u16)[fn_index(W, is_v)])


def unpack_codes(code_bytes, W, bits, is_v):
    byte, shift = code_position(W, bits, is_v)
    b = np.asarray(code_bytes, np.uint8)
    return ((b[byte] >> shift) & ((1 << bits) - 1)).astype(np.uint8)


def parse_ledger_block(blk, W, bits):
    """One (slot, head) ledger block -> codes_k [W][D], codes_v, s_k [D], m_k, s_v [W], m_v (fp16)."""
    blk = np.asarray(blk, np.uint8)
    cb = W * D * bits // 8
    ks = blk[2 * cb:2 * cb + 2 * D].view(np.float16)
    km = blk[2 * cb + 2 * D:2 * cb + 4 * D].view(np.float16)
    vs = blk[2 * cb + 4 * D:2 * cb + 4 * D + 2 * W].view(np.float16)
    vm = blk[2 * cb + 4 * D + 2 * W:2 * cb + 4 * D + 4 * W].view(np.float16)
    return (unpack_codes(blk[:cb], W, bits, False), unpack_codes(blk[cb:2 * cb], W, bits, True), ks, km, vs, vm)


def pack_block(values_f32, W, is_v):
    """[W][D] bf16-valued float32 -> [W*D] uint16 fragment-native block (inverse of unpack_block)."""
    u = (np.asarray(values_f32, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    out = np.zeros(W * D, np.uint16)
    out[fn_index(W, is_v)] = u
    return out
