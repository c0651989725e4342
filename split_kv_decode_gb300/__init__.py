"""Split-KV (flash-decoding) decode attention for GB300 (sm_103a)."""
