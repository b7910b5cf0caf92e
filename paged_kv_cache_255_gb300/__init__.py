"""libpagedattn: paged KV-cache store and single-token decode attention for GB300."""
