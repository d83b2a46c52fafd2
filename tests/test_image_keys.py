"""Image keys for the radix tree ("SGLang: Efficient Execution of Structured
Language Model Programs", unite.ai, es, "SGLang: Evaluación y resultados",
multimodal results: the hash of an input image is its key in the radix tree).

The oracle (oracle/keys.py) is pinned by the published test vectors of its two
building blocks; the native rx_image_keys must match it bit for bit, and the
keys must let requests about the same image share a cached prefix."""
import numpy as np
import pytest

from oracle import keys as ref
from oracle.tree_ref import RadixTreeRef
from prefix_shared_kv_radixattention_gb300 import binding as rx


def test_fnv1a64_published_vectors():
    """Test vectors of the FNV-1a 64-bit hash from its specification
    (Fowler, Noll, Vo): the empty input gives the offset basis."""
    assert ref.fnv1a64(b"") == 0xCBF29CE484222325
    assert ref.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert ref.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_splitmix64_published_outputs():
    """The first outputs of SplitMix64 (Steele, Lea, Flood; Vigna's reference
    code) from seed 0."""
    assert ref.splitmix64(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_oracle_keys_shape():
    k = ref.image_keys(b"pixels", 5)
    assert len(k) == 5 and all(x < 0 for x in k) and len(set(k)) == 5
    seeds = ref.splitmix64(ref.fnv1a64(b"pixels"), 5)
    assert [x & ((1 << 63) - 1) for x in k] == [s & ((1 << 63) - 1) for s in seeds]
    assert ref.image_keys(b"", 0) == []


@pytest.mark.parametrize("seed", range(8))
def test_native_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    data = rng.integers(0, 256, size=int(rng.integers(0, 5000)), dtype=np.uint8).tobytes()
    n = int(rng.integers(0, 700))
    assert rx.rx_image_keys(data, n).tolist() == ref.image_keys(data, n)


def test_keys_separate_images():
    a = bytes(range(256)) * 4
    b = bytearray(a)
    b[513] ^= 1                       # one bit differs
    ka, kb = rx.rx_image_keys(a, 64), rx.rx_image_keys(bytes(b), 64)
    assert rx.rx_image_keys(a, 64).tolist() == ka.tolist()
    assert not set(ka.tolist()) & set(kb.tolist())
    assert (ka < 0).all() and (kb < 0).all()


def test_requests_about_one_image_share_its_tokens():
    """text + image + text: a second request with the same system text and
    image matches through the image; one with another image stops at the
    text before it.  Native tree and oracle trie agree."""
    sys_text = list(range(100, 140))
    img_a, img_b = b"\x01\x02" * 3000, b"\x01\x02" * 2999 + b"\x01\x03"
    ka = rx.rx_image_keys(img_a, 576).tolist()
    kb = rx.rx_image_keys(img_b, 576).tolist()
    first = sys_text + ka + [7, 8, 9]
    same = sys_text + ka + [5, 6]
    other = sys_text + kb + [7, 8, 9]
    nat, oracle_t = rx.RadixTree(), RadixTreeRef()
    nat.insert(first, list(range(len(first))))
    oracle_t.insert(first, list(range(len(first))))
    for req, want in ((same, len(sys_text) + 576), (other, len(sys_text))):
        assert nat.prefix_len(req) == oracle_t.prefix_len(req) == want


def test_invalid_arguments():
    lib = rx.library()
    assert lib.rx_image_keys(None, 4, 1, None) == rx.RX_ERR_INVALID
    assert lib.rx_image_keys(None, 0, -1, None) == rx.RX_ERR_INVALID
    assert lib.rx_image_keys(None, 0, 0, None) == rx.RX_OK
