"""libexpzip: lossless BF16 exponent codecs on sm_103a (package marker; see binding)."""
